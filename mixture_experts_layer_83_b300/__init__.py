"""B300 (sm_103a) forward pass of one sparse Mixture-of-Experts FFN layer.

A thin ctypes binding of ``libmoe_b300.so`` with the same entry points as the C ABI in
``include/moe_layer.h``.  Every function only marshals arguments: each step of the layer runs
in the library's CUDA kernels.  Array arguments may be torch tensors (their ``data_ptr()`` is
passed) or raw device addresses (ints).  There is no fallback: if the library is missing the
first call raises.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_SCORE_SOFTMAX = 0
MOE_SCORE_SIGMOID = 1
MOE_DTYPE_F32 = 0
MOE_DTYPE_BF16 = 1
MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE = -5
MOE_NUM_STAGE_EVENTS = 8
STAGE_NAMES = ("router_gemm", "topk", "dispatch", "gather", "gateup_gemm", "down_gemm", "combine")

EXPORTED = ("moe_layer_workspace_size", "moe_layer_forward", "moe_layer_forward_ex",
            "moe_route_from_keys", "moe_route_from_keys_grouped", "moe_route_from_keys_noalloc",
            "moe_debug_gemm_tiles", "moe_debug_unclustered_pair", "moe_debug_wait_timeout",
            "moe_eplb_plan", "moe_load_expectation", "moe_load_report",
            "moe_layer_num_launches", "moe_workspace_status", "moe_status_string",
            "moe_last_cuda_error_name", "moe_workspace_kernel_clocks")
MOE_NOALLOC_SCRATCH_BYTES = 1 << 20


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("F", ctypes.c_int), ("Fs", ctypes.c_int),
                ("dtype", ctypes.c_int)]


class MoeSharedExpert(ctypes.Structure):
    _fields_ = [("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p)]


class MoeForwardOpts(ctypes.Structure):
    _fields_ = [("stage_events", ctypes.POINTER(ctypes.c_void_p)), ("n_groups", ctypes.c_int),
                ("topk_groups", ctypes.c_int), ("capacity_factor", ctypes.c_double),
                ("dropped", ctypes.c_void_p), ("reroute", ctypes.c_int)]


class MoeError(RuntimeError):
    def __init__(self, code, what):
        detail = f", {moe_last_cuda_error_name()}" if code == MOE_ERR_CUDA else ""
        super().__init__(f"{what}: {moe_status_string(code)} ({code}{detail})")
        self.code = code


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} not found: build it with __graft_entry__.build()")
        l = ctypes.CDLL(LIB_PATH)
        vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        shp = ctypes.POINTER(MoeShape)
        l.moe_layer_workspace_size.argtypes = [shp]
        l.moe_layer_workspace_size.restype = sz
        fwd = [shp, vp, vp, vp, vp, ci, vp, ctypes.POINTER(MoeSharedExpert), vp, vp, vp, sz, vp,
               vp, vp, vp]
        l.moe_layer_forward.argtypes = fwd
        l.moe_layer_forward.restype = ci
        l.moe_layer_forward_ex.argtypes = fwd + [ctypes.POINTER(MoeForwardOpts)]
        l.moe_layer_forward_ex.restype = ci
        l.moe_route_from_keys.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        l.moe_route_from_keys.restype = ci
        l.moe_route_from_keys_grouped.argtypes = [shp, vp, vp, ci, ci, vp, vp, vp, vp, vp, vp, vp,
                                                  sz, vp]
        l.moe_route_from_keys_grouped.restype = ci
        l.moe_route_from_keys_noalloc.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        l.moe_route_from_keys_noalloc.restype = ci
        l.moe_debug_gemm_tiles.argtypes = [shp, ci, ci, vp, vp, ci, vp]
        l.moe_debug_gemm_tiles.restype = ci
        l.moe_debug_unclustered_pair.argtypes = [vp, vp]
        l.moe_debug_unclustered_pair.restype = ci
        l.moe_debug_wait_timeout.argtypes = [vp, ctypes.c_ulonglong, vp]
        l.moe_debug_wait_timeout.restype = ci
        l.moe_eplb_plan.argtypes = [vp, ci, ci, ci, vp, vp, vp]
        l.moe_eplb_plan.restype = ci
        dp = ctypes.POINTER(ctypes.c_double)
        l.moe_load_expectation.argtypes = [ci, ci, ci, ci, ci, dp, dp]
        l.moe_load_expectation.restype = ci
        l.moe_load_report.argtypes = [vp, ci, ci, vp]
        l.moe_load_report.restype = ci
        l.moe_layer_num_launches.argtypes = [shp]
        l.moe_layer_num_launches.restype = ci
        l.moe_workspace_status.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(ci)]
        l.moe_workspace_status.restype = ci
        l.moe_workspace_kernel_clocks.argtypes = [vp, vp]
        l.moe_workspace_kernel_clocks.restype = ci
        l.moe_last_cuda_error_name.argtypes = []
        l.moe_last_cuda_error_name.restype = ctypes.c_char_p
        l.moe_status_string.argtypes = [ci]
        l.moe_status_string.restype = ctypes.c_char_p
        _lib = l
    return _lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_shape(T, d, E, k, F, Fs=0, dtype=MOE_DTYPE_BF16):
    return MoeShape(T, d, E, k, F, Fs, dtype)


def moe_last_cuda_error_name():
    return lib().moe_last_cuda_error_name().decode()


def moe_status_string(code):
    return lib().moe_status_string(int(code)).decode()


def moe_layer_workspace_size(shape):
    return int(lib().moe_layer_workspace_size(ctypes.byref(shape)))


def moe_layer_num_launches(shape):
    return int(lib().moe_layer_num_launches(ctypes.byref(shape)))


def _shared(shared_expert):
    if shared_expert is None:
        return None
    gu, dn = shared_expert
    return ctypes.byref(MoeSharedExpert(_ptr(gu), _ptr(dn)))


def moe_layer_forward(shape, x, w_router, w_gate_up, w_down, score_fn, bias, shared_expert,
                      out, expert_counts, workspace, workspace_bytes=None, stream=None,
                      topk_idx_out=None, topk_w_out=None, sorted_token_out=None,
                      stage_events=None, n_groups=0, topk_groups=0, capacity_factor=0.0,
                      dropped=None, reroute=0, check=True):
    """One forward pass; ``shared_expert`` is None or (w_gate_up, w_down); ``n_groups`` /
    ``topk_groups`` select group-limited routing (0 / 0: plain top-k); ``capacity_factor`` > 0
    caps each expert's assignments (``dropped``: optional device int receiving the number
    dropped); ``reroute`` > 0 (with a capacity) moves overflow to each token's next-best
    experts instead of dropping it.  Returns the status (raises MoeError on failure when
    ``check``)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args = [ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(w_gate_up), _ptr(w_down),
            int(score_fn), _ptr(bias), _shared(shared_expert), _ptr(out), _ptr(expert_counts),
            _ptr(workspace), int(workspace_bytes), _stream(stream), _ptr(topk_idx_out),
            _ptr(topk_w_out), _ptr(sorted_token_out)]
    if stage_events is None and n_groups == 0 and topk_groups == 0 and capacity_factor == 0 \
            and dropped is None and reroute == 0:
        rc = lib().moe_layer_forward(*args)
    else:
        arr = None
        if stage_events is not None:
            for e in stage_events:
                if not e.cuda_event:   # torch creates the CUDA event on its first record
                    e.record()
            arr = (ctypes.c_void_p * MOE_NUM_STAGE_EVENTS)(*[e.cuda_event for e in stage_events])
        opts = MoeForwardOpts(arr, int(n_groups), int(topk_groups), float(capacity_factor),
                              _ptr(dropped), int(reroute))
        rc = lib().moe_layer_forward_ex(*args, ctypes.byref(opts))
    if check and rc != MOE_OK:
        raise MoeError(rc, "moe_layer_forward")
    return rc


moe_layer_forward_ex = moe_layer_forward


def moe_route_from_keys(shape, sel_key, gate_score, topk_idx, topk_w, expert_counts,
                        expert_offsets, sorted_token, slot_pos, workspace, workspace_bytes=None,
                        stream=None, check=True):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib().moe_route_from_keys(ctypes.byref(shape), _ptr(sel_key), _ptr(gate_score),
                                   _ptr(topk_idx), _ptr(topk_w), _ptr(expert_counts),
                                   _ptr(expert_offsets), _ptr(sorted_token), _ptr(slot_pos),
                                   _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check and rc != MOE_OK:
        raise MoeError(rc, "moe_route_from_keys")
    return rc


def moe_route_from_keys_grouped(shape, sel_key, gate_score, n_groups, topk_groups, topk_idx,
                                topk_w, expert_counts, expert_offsets, sorted_token, slot_pos,
                                workspace, workspace_bytes=None, stream=None, check=True):
    """moe_route_from_keys with group-limited routing (see include/moe_layer.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib().moe_route_from_keys_grouped(ctypes.byref(shape), _ptr(sel_key), _ptr(gate_score),
                                           int(n_groups), int(topk_groups), _ptr(topk_idx),
                                           _ptr(topk_w), _ptr(expert_counts),
                                           _ptr(expert_offsets), _ptr(sorted_token),
                                           _ptr(slot_pos), _ptr(workspace), int(workspace_bytes),
                                           _stream(stream))
    if check and rc != MOE_OK:
        raise MoeError(rc, "moe_route_from_keys_grouped")
    return rc


def moe_route_from_keys_noalloc(shape, sel_key, gate_score, topk_idx, topk_w, expert_counts,
                                expert_offsets, sorted_token, slot_pos, stream=None, check=True):
    """moe_route_from_keys without a workspace, for callers that cannot allocate device memory:
    the scratch is a fixed array inside the library (see include/moe_layer.h)."""
    rc = lib().moe_route_from_keys_noalloc(ctypes.byref(shape), _ptr(sel_key), _ptr(gate_score),
                                           _ptr(topk_idx), _ptr(topk_w), _ptr(expert_counts),
                                           _ptr(expert_offsets), _ptr(sorted_token),
                                           _ptr(slot_pos), _stream(stream))
    if check and rc != MOE_OK:
        raise MoeError(rc, "moe_route_from_keys_noalloc")
    return rc


def moe_debug_gemm_tiles(shape, which, expert_counts=None, num_sms=148):
    """Host-side tile schedule of GEMM ``which`` (0 router, 1 gate/up, 2 down): returns
    (tiles [n][7] int32 numpy array, geometry dict)."""
    import numpy as np
    counts = None if expert_counts is None else np.ascontiguousarray(expert_counts, np.int32)
    geo = np.zeros(9, dtype=np.int32)
    n = lib().moe_debug_gemm_tiles(ctypes.byref(shape), which, num_sms,
                                   None if counts is None else counts.ctypes.data, None, 0,
                                   geo.ctypes.data)
    if n < 0:
        raise MoeError(n, "moe_debug_gemm_tiles")
    tiles = np.zeros((max(n, 1), 7), dtype=np.int32)
    lib().moe_debug_gemm_tiles(ctypes.byref(shape), which, num_sms,
                               None if counts is None else counts.ctypes.data, tiles.ctypes.data,
                               n, geo.ctypes.data)
    keys = ("bn", "stages_a", "stages_b", "smem_bytes", "m_tiles0", "m_tiles1", "group", "K0",
            "cg")
    return tiles[:n], dict(zip(keys, (int(v) for v in geo)))


def moe_debug_unclustered_pair(workspace, stream=None, check=True):
    """Launch the CTA-pair GEMM without clusters (it records device code 5 and returns)."""
    rc = lib().moe_debug_unclustered_pair(_ptr(workspace), _stream(stream))
    if check and rc != MOE_OK:
        raise MoeError(rc, "moe_debug_unclustered_pair")
    return rc


def moe_debug_wait_timeout(workspace, limit_ns, stream=None, check=True):
    """Launch a wait that nothing completes, limited to ``limit_ns`` (records device code 6)."""
    rc = lib().moe_debug_wait_timeout(_ptr(workspace), int(limit_ns), _stream(stream))
    if check and rc != MOE_OK:
        raise MoeError(rc, "moe_debug_wait_timeout")
    return rc


def moe_eplb_plan(expert_load, n_gpus, n_redundant=0):
    """Redundant-expert placement plan (host): returns (slot_expert [S] int32, slot_gpu [S]
    int32, gpu_load [n_gpus] float64), S = E + n_redundant."""
    import numpy as np
    load = np.ascontiguousarray(expert_load, np.int32)
    S = load.size + int(n_redundant)
    se = np.zeros(max(S, 1), np.int32)
    sg = np.zeros(max(S, 1), np.int32)
    gl = np.zeros(max(int(n_gpus), 1), np.float64)
    rc = lib().moe_eplb_plan(load.ctypes.data, load.size, int(n_gpus), int(n_redundant),
                             se.ctypes.data, sg.ctypes.data, gl.ctypes.data)
    if rc != MOE_OK:
        raise MoeError(rc, "moe_eplb_plan")
    return se[:S], sg[:S], gl[:int(n_gpus)]


def moe_load_expectation(tokens_per_gpu, E, k, n_gpus=1, n_redundant=0):
    """(expert slots per GPU, expected rows per expert) under uniform routing (host)."""
    slots, tpe = ctypes.c_double(0), ctypes.c_double(0)
    rc = lib().moe_load_expectation(int(tokens_per_gpu), int(E), int(k), int(n_gpus),
                                    int(n_redundant), ctypes.byref(slots), ctypes.byref(tpe))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_load_expectation")
    return slots.value, tpe.value


def moe_load_report(expert_counts, n_groups=1):
    """Load statistics of host expert counts: dict with mean rows per expert, max/mean over
    experts, max/mean over n_groups contiguous groups and the experts touched."""
    import numpy as np
    counts = np.ascontiguousarray(expert_counts, np.int32)
    rep = np.zeros(4, np.float64)
    rc = lib().moe_load_report(counts.ctypes.data, counts.size, int(n_groups), rep.ctypes.data)
    if rc != MOE_OK:
        raise MoeError(rc, "moe_load_report")
    return {"mean_rows_per_expert": float(rep[0]), "expert_max_over_mean": float(rep[1]),
            "group_max_over_mean": float(rep[2]), "experts_touched": int(rep[3])}


def moe_workspace_kernel_clocks(workspace):
    """{kernel: (SM MHz, ms)} of CTA 0 of the router, gate/up and down tensor-core kernels of
    the latest forward pass on this workspace (synchronous)."""
    import numpy as np
    rep = np.zeros(6, np.float64)
    rc = lib().moe_workspace_kernel_clocks(_ptr(workspace), rep.ctypes.data)
    if rc != MOE_OK:
        raise MoeError(rc, "moe_workspace_kernel_clocks")
    return {name: (float(rep[2 * i]), float(rep[2 * i + 1]))
            for i, name in enumerate(("router", "gateup_gemm", "down_gemm"))}


def moe_workspace_status(workspace):
    """(status, detail) of a workspace's device status word (synchronous)."""
    st, det = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().moe_workspace_status(_ptr(workspace), ctypes.byref(st), ctypes.byref(det))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_workspace_status")
    return st.value, det.value
