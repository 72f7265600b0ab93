"""Seeded random weights and prompts.

Procedure (one generator per model, tensors drawn in a fixed order):
``rng = numpy.random.default_rng(seed)``; for each tensor in ``TENSOR_ORDER``
draw ``rng.standard_normal(shape, float32) * 0.02`` and store it as bf16
(round-to-nearest-even on the fp32 bit pattern) or as IEEE fp16.  RMSNorm
gains are exactly 1.  Prompt ids are uniform over the vocabulary from
``default_rng([seed, 1])``.
"""
import numpy as np

from .configs import Workload

# Draw order.  Per layer: q, k, v, o, gate, up, down.
LAYER_TENSORS = ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown")
TENSOR_ORDER = ("embed",) + tuple(f"layer.{t}" for t in LAYER_TENSORS) + ("lm_head",)


def tensor_shape(w: Workload, name: str):
    d, qd, kd, f, v = w.d_model, w.q_dim, w.kv_dim, w.d_ffn, w.vocab
    return {
        "embed": (v, d), "lm_head": (v, d),
        "wq": (qd, d), "wk": (kd, d), "wv": (kd, d), "wo": (d, qd),
        "wgate": (f, d), "wup": (f, d), "wdown": (d, f),
    }[name]


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Storage conversion fp32 -> bf16 bits, round to nearest even (finite input)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (u >> np.uint32(16)).astype(np.uint16)


def _store(a: np.ndarray, base_dtype: str) -> np.ndarray:
    if base_dtype == "bf16":
        return _f32_to_bf16_bits(a)
    if base_dtype == "fp16":
        return a.astype(np.float16).view(np.uint16)
    raise ValueError(base_dtype)


def bits_to_f32(bits: np.ndarray, base_dtype: str) -> np.ndarray:
    """Exact widening of stored bf16 / fp16 bit patterns to float32."""
    if base_dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if base_dtype == "fp16":
        return bits.view(np.float16).astype(np.float32)
    raise ValueError(base_dtype)


def generate_weights(w: Workload) -> dict:
    """Return {name: uint16 bit array} for every tensor plus norm gains.

    Keys: ``embed``, ``lm_head``, ``final_norm``, and per layer ``l{i}.wq`` ...
    ``l{i}.wdown``, ``l{i}.attn_norm``, ``l{i}.ffn_norm``.  All arrays hold
    bf16 or fp16 bit patterns as given by ``w.base_dtype``.
    """
    rng = np.random.default_rng(w.seed)
    scale = np.float32(0.02)
    out = {}

    def draw(shape):
        a = rng.standard_normal(shape, dtype=np.float32)
        a *= scale
        return _store(a, w.base_dtype)

    out["embed"] = draw(tensor_shape(w, "embed"))
    for i in range(w.n_layers):
        for t in LAYER_TENSORS:
            out[f"l{i}.{t}"] = draw(tensor_shape(w, t))
    out["lm_head"] = draw(tensor_shape(w, "lm_head"))
    one = _store(np.ones(w.d_model, np.float32), w.base_dtype)
    for i in range(w.n_layers):
        out[f"l{i}.attn_norm"] = one.copy()
        out[f"l{i}.ffn_norm"] = one.copy()
    out["final_norm"] = one.copy()
    return out


def generate_prompt(w: Workload, n: int = None) -> np.ndarray:
    n = w.prompt_len if n is None else n
    return np.random.default_rng([w.seed, 1]).integers(0, w.vocab, n, dtype=np.int32)


def random_tokens(w: Workload, n: int, stream: int) -> np.ndarray:
    """Extra uniform token streams (teacher-forcing inputs in tests)."""
    return np.random.default_rng([w.seed, 2, stream]).integers(0, w.vocab, n, dtype=np.int32)
