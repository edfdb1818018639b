"""Named synthetic workloads for one sparse MoE FFN layer.

Each entry fixes the layer shape, the score function, the element type and the seed of
the counter-based generator in ``moe_inputs.host`` / ``moe_inputs.device``.  Nothing here
computes any part of the layer; it only describes the inputs.

Shapes follow the model families the pages name: "Expert-Parallel MoE Inference: Serving
Sparse Models at Scale" (Context and Background: top-k of 128 or 256 experts) and
"Tensor vs Expert vs Data Parallelism for MoE Serving" (Context and Background: 256 routed
experts plus one shared expert and top-8; Communication volume: hidden size 7,168).
"""

# Tensor ids of the counter-based generator (part of the input recipe).
TID_X = 1
TID_W_ROUTER = 2
TID_W_GATE_UP = 3
TID_W_DOWN = 4
TID_BIAS = 5
TID_SH_GATE_UP = 6
TID_SH_DOWN = 7
TID_ZIPF_PERM = 8

SOFTMAX = 0
SIGMOID = 1

CONFIGS = {
    0: dict(name="tiny-fp32", T=64, d=128, E=8, k=2, F=256, Fs=0, dtype="f32",
            score=SOFTMAX, bias_range=0.0, zipf=None, groups=0, seed=0),
    1: dict(name="mixtral-8x7b-prefill", T=4096, d=4096, E=8, k=2, F=14336, Fs=0, dtype="bf16",
            score=SOFTMAX, bias_range=0.0, zipf=None, groups=0, seed=1),
    2: dict(name="deepseek-v3-prefill", T=8192, d=7168, E=256, k=8, F=2048, Fs=2048, dtype="bf16",
            score=SIGMOID, bias_range=0.01, zipf=None, groups=0, seed=2),
    3: dict(name="deepseek-v3-decode", T=128, d=7168, E=256, k=8, F=2048, Fs=2048, dtype="bf16",
            score=SIGMOID, bias_range=0.01, zipf=None, groups=0, seed=3),
    4: dict(name="zipf-skewed", T=16384, d=4096, E=128, k=8, F=1536, Fs=0, dtype="bf16",
            score=SOFTMAX, bias_range=0.0, zipf=dict(s=1.2, scale=2.0), groups=8, seed=4),
}


def make_shape(T, d, E, k, F, Fs=0, dtype="bf16", score=SOFTMAX, bias_range=0.0, zipf=None,
               groups=0, seed=0, name="custom"):
    """A workload dict with the same keys as the named ones (used for test sizes)."""
    return dict(name=name, T=T, d=d, E=E, k=k, F=F, Fs=Fs, dtype=dtype, score=score,
                bias_range=bias_range, zipf=zipf, groups=groups, seed=seed)


def get(cfg):
    if isinstance(cfg, dict):
        return cfg
    return CONFIGS[int(cfg)]
