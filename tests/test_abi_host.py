"""C ABI checks that need no GPU: exported symbols, argument validation (all decided on the
host before anything is enqueued), workspace sizing and the grouped-GEMM tile schedule
(computed by the library's own decoder, the code the kernel runs)."""
import ctypes
import os
import re

import numpy as np
import pytest

import mixture_experts_layer_83_b300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_layer.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 8
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.EXPORTED) == names


def shape(T=64, d=128, E=8, k=2, F=128, Fs=0, dtype=moe.MOE_DTYPE_BF16):
    return moe.make_shape(T, d, E, k, F, Fs, dtype)


@pytest.mark.parametrize("bad", [dict(T=0), dict(E=0), dict(k=0), dict(k=9), dict(k=33, E=64),
                                 dict(E=1025, k=2), dict(d=0), dict(F=0), dict(Fs=-1),
                                 dict(dtype=7)])
def test_workspace_size_rejects_invalid_shapes(bad):
    assert moe.moe_layer_workspace_size(shape(**bad)) == 0


def test_workspace_size_grows_with_the_problem():
    a = moe.moe_layer_workspace_size(shape())
    b = moe.moe_layer_workspace_size(shape(T=128))
    c = moe.moe_layer_workspace_size(shape(Fs=64))
    f = moe.moe_layer_workspace_size(shape(dtype=moe.MOE_DTYPE_F32))
    assert 0 < a < b and a < c and a < f
    R, d, F = 64 * 2, 128, 128
    assert a >= R * d * 2 + R * F * 2 + 64 * 8 * 4


def _forward(s, ptrs=None, ws_bytes=1 << 40, **kw):
    p = dict(x=16, w_router=16, w_gate_up=16, w_down=16, out=16, expert_counts=16,
             workspace=16, bias=None, shared=None)
    p.update(ptrs or {})
    return moe.moe_layer_forward(s, p["x"], p["w_router"], p["w_gate_up"], p["w_down"],
                                 kw.get("score", moe.MOE_SCORE_SOFTMAX), p["bias"], p["shared"],
                                 p["out"], p["expert_counts"], p["workspace"], ws_bytes, stream=0,
                                 check=False)


@pytest.mark.parametrize("field", ["x", "w_router", "w_gate_up", "w_down", "out", "expert_counts",
                                   "workspace"])
def test_forward_rejects_null_pointers(field):
    assert _forward(shape(), {field: None}) == moe.MOE_ERR_INVALID_ARG


def test_forward_rejects_misaligned_pointers():
    assert _forward(shape(), {"x": 18}) == moe.MOE_ERR_INVALID_ARG
    assert _forward(shape(), {"bias": 20}) == moe.MOE_ERR_INVALID_ARG


def test_forward_rejects_bad_score_fn_and_shared_expert_mismatch():
    assert _forward(shape(), score=3) == moe.MOE_ERR_INVALID_ARG
    assert _forward(shape(Fs=64)) == moe.MOE_ERR_INVALID_ARG            # shared weights missing
    assert _forward(shape(), {"shared": (16, 16)}) == moe.MOE_ERR_INVALID_ARG  # Fs == 0
    assert _forward(shape(Fs=64), {"shared": (16, None)}) == moe.MOE_ERR_INVALID_ARG


def test_forward_rejects_shapes_the_tensor_core_path_does_not_take():
    assert _forward(shape(d=100)) == moe.MOE_ERR_UNSUPPORTED
    assert _forward(shape(F=96)) == moe.MOE_ERR_UNSUPPORTED
    assert _forward(shape(Fs=32), {"shared": (16, 16)}) == moe.MOE_ERR_UNSUPPORTED


def test_forward_rejects_a_small_workspace():
    s = shape()
    need = moe.moe_layer_workspace_size(s)
    assert _forward(s, ws_bytes=need - 1) == moe.MOE_ERR_WORKSPACE


def test_route_from_keys_argument_checks():
    s = shape()
    args = [16] * 8   # fake addresses: every call below must be rejected before any launch
    bad = list(args)
    bad[2] = None
    assert moe.moe_route_from_keys(s, *bad, 16, 1 << 30, stream=0,
                                   check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_route_from_keys(shape(k=9), *args, 16, 1 << 30, stream=0,
                                   check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_route_from_keys(s, *args, 16, 64, stream=0,
                                   check=False) == moe.MOE_ERR_WORKSPACE


def test_status_strings_and_launch_count():
    assert moe.moe_status_string(0) == "ok"
    assert "workspace" in moe.moe_status_string(moe.MOE_ERR_WORKSPACE)
    # bf16 with up to 256 experts: one fused router launch (gate GEMM + top-k); decode-sized
    # segments: the gate/up GEMM gathers its token rows (no gather launch); long segments and
    # the fp32 layer run the separate row gather; more than 256 experts: router GEMM + top-k
    assert moe.moe_layer_num_launches(shape()) == 7
    assert moe.moe_layer_num_launches(shape(T=4096)) == 8
    assert moe.moe_layer_num_launches(shape(T=65536, E=512)) == 9
    assert moe.moe_layer_num_launches(shape(dtype=moe.MOE_DTYPE_F32)) == 9
    assert moe.moe_layer_num_launches(shape(T=0)) == -1


# ------------------------------------------------------------------ tile schedule
def _check_schedule(s, which, counts):
    tiles, geo = moe.moe_debug_gemm_tiles(s, which, counts)
    assert 2 <= geo["stages_a"] <= 12 and 2 <= geo["stages_b"] <= 8
    assert geo["cg"] == (1 if which == 0 else 2)
    # one-CTA and wide-pair GEMMs may use the 227 KiB opt-in; narrow pair CTAs (experts
    # averaging at most 64 rows) share their SM with a second one
    narrow = which > 0 and -(-s.T * s.k // s.E) <= 64
    assert geo["smem_bytes"] <= (114688 if narrow else 232448)
    bn = geo["bn"]
    # the expert GEMMs run on wide CTA pairs for long segments (n-tiles up to 384 token rows),
    # the router up to 256
    assert bn % 16 == 0 and 16 <= bn <= (384 if which > 0 else 256)
    if which == 0:
        seg_rows = [s.T]
        seg_off = [0, s.T]
        m_tiles = [(s.E + 127) // 128]
    else:
        seg_rows = list(counts)
        seg_off = np.concatenate([[0], np.cumsum(counts)])
        m_tiles = [geo["m_tiles0"], geo["m_tiles1"]]
    covered = {}
    for prob, seg, m, row0, ncols, valid, box1 in tiles.tolist():
        assert ncols % 16 == 0 and 16 <= ncols <= bn
        assert 1 <= valid <= ncols
        assert 0 <= m < m_tiles[prob]
        if prob == 0:
            lo, hi = seg_off[seg], seg_off[seg + 1]
        else:
            lo, hi = 0, s.T
        assert lo <= row0 and row0 + valid <= hi
        assert row0 + valid == hi or valid == ncols
        for r in range(row0, row0 + valid):
            key = (prob, seg, m, r)
            assert key not in covered, key
            covered[key] = 1
        if which == 2:   # down: second box only while inside the d rows of the expert
            assert box1 == (m * 128 + 64 < s.d)
        elif which == 1:
            assert box1 == 1
        else:
            assert box1 == (s.E >= 64 and m * 128 + 64 < s.E)
    want = sum(m_tiles[0] * n for n in seg_rows)
    if which > 0 and s.Fs > 0:
        want += m_tiles[1] * s.T
    assert len(covered) == want
    if geo["cg"] == 2:
        # the CTAs of a pair share the token rows: tile 2j is listed with its partner 2j + 1
        # right after it, unless 2j + 1 is past the weight rows
        t = tiles.tolist()
        i = 0
        while i < len(t):
            prob, seg, m, row0, ncols = t[i][:5]
            assert m % 2 == 0
            if m + 1 < m_tiles[prob]:
                assert t[i + 1][:5] == [prob, seg, m + 1, row0, ncols]
                i += 2
            else:
                i += 1


@pytest.mark.parametrize("which", [1, 2])
@pytest.mark.parametrize("case", ["uniform", "ragged", "one_hot", "decode", "shared", "long",
                                  "long_skewed"])
def test_expert_gemm_schedule_covers_every_row_once(which, case):
    rng = np.random.default_rng(["uniform", "ragged", "one_hot", "decode", "shared", "long",
                                 "long_skewed"].index(case) * 10 + which)
    if case == "uniform":
        s = shape(T=512, d=256, E=16, k=4, F=192)
        counts = np.full(16, 512 * 4 // 16)
    elif case == "ragged":
        s = shape(T=700, d=320, E=24, k=3, F=128)
        counts = rng.multinomial(700 * 3, np.ones(24) / 24)
        counts[3] = counts[3] + counts[5]
        counts[5] = 0
    elif case == "one_hot":
        s = shape(T=1000, d=128, E=8, k=1, F=64)
        counts = np.zeros(8, dtype=int)
        counts[6] = 1000
    elif case == "decode":
        s = shape(T=128, d=7168, E=256, k=8, F=2048, Fs=2048)
        counts = rng.multinomial(128 * 8, np.ones(256) / 256)
    elif case == "long":    # experts average 512 rows: every tile tall
        s = shape(T=2048, d=256, E=8, k=2, F=256)
        counts = rng.multinomial(2048 * 2, np.ones(8) / 8)
    elif case == "long_skewed":
        s = shape(T=3000, d=512, E=16, k=2, F=128, Fs=64)
        w = 1.0 / np.arange(1, 17) ** 1.2
        counts = rng.multinomial(3000 * 2, w / w.sum())
        counts[9] = 0
    else:
        s = shape(T=333, d=192, E=5, k=2, F=64, Fs=128)
        counts = rng.multinomial(333 * 2, np.ones(5) / 5)
    _check_schedule(s, which, counts)


@pytest.mark.parametrize("which", [1, 2])
def test_long_segments_run_as_tall_tiles(which):
    """Experts averaging 384 rows or more: every segment runs as ceil(rows / 256) tall n-tiles
    (two scheduled weight tiles, i.e. four 128-row CTA tiles, over the same token rows), rows
    split evenly in 16-row units."""
    s = shape(T=2048, d=256, E=8, k=2, F=256)
    counts = np.array([700, 256, 257, 0, 1, 1000, 900, 981])
    tiles, geo = moe.moe_debug_gemm_tiles(s, which, counts)
    assert geo["bn"] == 256
    m_cta = geo["m_tiles0"]
    off = np.concatenate([[0], np.cumsum(counts)])
    for e, n in enumerate(counts):
        t = tiles[(tiles[:, 0] == 0) & (tiles[:, 1] == e)]
        if n == 0:
            assert len(t) == 0
            continue
        nt = -(-n // 256)
        starts = sorted(set(t[:, 3].tolist()))
        assert len(starts) == nt and starts[0] == off[e]
        units = -(-n // 16)
        sizes = [16 * (units // nt + (j < units % nt)) for j in range(nt)]
        assert sorted(set(t[:, 4].tolist())) == sorted(set(sizes))
        for r0 in starts:   # each n-tile meets every 128-row weight tile once
            assert sorted(t[t[:, 3] == r0][:, 2].tolist()) == list(range(m_cta))


@pytest.mark.parametrize("T,E", [(1, 8), (37, 8), (300, 100), (8192, 256), (128, 256), (64, 1)])
def test_router_gemm_schedule_covers_every_row_once(T, E):
    _check_schedule(shape(T=T, E=E, k=1, d=256), 0, None)


def test_prefill_geometry_uses_full_width_tiles():
    s = shape(T=8192, d=7168, E=256, k=8, F=2048, Fs=2048)
    _, geo = moe.moe_debug_gemm_tiles(s, 1, np.full(256, 256))
    # stage counts are multiples of the producer threads per ring (2 weight, 4 token producers
    # for the wide gate/up pairs; 2 and 2 for the down pairs)
    assert geo["bn"] == 384 and geo["stages_a"] == 6 and geo["stages_b"] == 4
    assert geo["m_tiles0"] == 32 and geo["cg"] == 2
    _, geo = moe.moe_debug_gemm_tiles(s, 2, np.full(256, 256))
    assert geo["bn"] == 384 and geo["stages_a"] == 6 and geo["stages_b"] == 4
    assert geo["m_tiles0"] == 56 and geo["cg"] == 2
    _, geo = moe.moe_debug_gemm_tiles(shape(T=128, d=7168, E=256, k=8, F=2048, Fs=2048), 1,
                                      np.full(256, 4))
    # decode-sized segments: gate/up on narrow pairs (two per TPC, 112 KiB each)
    assert geo["bn"] == 32 and geo["stages_a"] == 4 and geo["stages_b"] == 8


@pytest.mark.parametrize("which,m_tiles", [(1, 32), (2, 56)])
def test_prefill_expert_gemms_tall_and_wide_tiles(which, m_tiles):
    """Prefill expert GEMMs: segments of up to 256 rows run as tall tiles (four weight tiles of
    128 rows, i.e. two pairs, over all the segment's rows); longer ones as wide tiles (one pair
    over up to 384 rows)."""
    s = shape(T=8192, d=7168, E=256, k=8, F=2048, Fs=2048)
    counts = np.full(256, 256)
    counts[1] = 300
    counts[2] = 0
    counts[3] = 10
    tiles, geo = moe.moe_debug_gemm_tiles(s, which, counts)
    assert geo["m_tiles0"] == m_tiles
    routed = tiles[tiles[:, 0] == 0]
    for e, n in ((0, 256), (1, 300), (3, 10)):
        t = routed[routed[:, 1] == e]
        assert len(t) == m_tiles and sorted(t[:, 2].tolist()) == list(range(m_tiles))
        assert (t[:, 5] == n).all() and (t[:, 4] == (n + 15) // 16 * 16).all()
        if n <= 256:   # tall: the CTA tiles of one tile are four consecutive weight tiles
            assert (t[:, 2].reshape(-1, 4) == t[::4, 2:3] + np.arange(4)).all()
        else:          # wide: two consecutive weight tiles (a pair)
            assert (t[:, 2].reshape(-1, 2) == t[::2, 2:3] + np.arange(2)).all()
    assert (routed[:, 1] != 2).all()


def test_group_limited_routing_arguments_are_checked_before_launch():
    """Invalid group options are rejected on the host (fake pointers never reach a kernel)."""
    s = shape(T=16, E=64, k=8)
    args = [16] * 8
    for G, M in ((3, 1), (0, 1), (64, 1), (8, 0), (8, 9), (8, 1), (33, 2)):
        # (8, 1): 1 group of 8 experts holds exactly k = 8 -> allowed; every other case invalid
        rc = moe.moe_route_from_keys_grouped(s, 16, 16, G, M, *args[:6], 16, 1 << 30, stream=0,
                                             check=False) if (G, M) != (8, 1) else None
        if rc is not None:
            assert rc == moe.MOE_ERR_INVALID_ARG, (G, M, rc)
    s2 = shape(T=16, E=64, k=9)
    assert moe.moe_route_from_keys_grouped(s2, 16, 16, 8, 1, *args[:6], 16, 1 << 30, stream=0,
                                           check=False) == moe.MOE_ERR_INVALID_ARG


def test_error_path_diagnostics_check_arguments_before_launching():
    """The two device error-path diagnostics reject a null or misaligned workspace and a wait
    limit outside 1 us .. 1 s on the host, before anything is enqueued."""
    assert moe.moe_debug_unclustered_pair(None, stream=0, check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_debug_unclustered_pair(20, stream=0, check=False) == moe.MOE_ERR_INVALID_ARG
    for ws, limit in ((None, 10_000), (20, 10_000), (256, 999), (256, 1_000_000_001)):
        assert moe.moe_debug_wait_timeout(ws, limit, stream=0, check=False) == \
            moe.MOE_ERR_INVALID_ARG


def test_reroute_option_checked_before_launching():
    """Rerouting needs a capacity, at most 32 candidates per token and no more than E; the
    checks run on the host before anything is enqueued."""
    for kw in (dict(reroute=2), dict(capacity_factor=1.0, reroute=-1),
               dict(capacity_factor=1.0, reroute=7), dict(capacity_factor=1.0, reroute=31),
               # 2 of 4 groups keep 4 of the 8 experts: 2 + 3 candidates do not fit
               dict(capacity_factor=1.0, reroute=3, n_groups=4, topk_groups=2)):
        rc = moe.moe_layer_forward(shape(), 16, 16, 16, 16, moe.MOE_SCORE_SOFTMAX, None, None, 16,
                                   16, 16, 1 << 40, stream=0, check=False, **kw)
        assert rc == moe.MOE_ERR_INVALID_ARG, kw
