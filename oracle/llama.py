"""Reference forward pass of a Llama-style decoder (float64, CPU).

Each function states the step it writes out.  Definitions follow the standard
Llama decoder that the AutoMegaKernel explainer ("Methodology": compiles
HuggingFace Llama-family models; "Results": greedy decode must match token for
token) and the Kog monokernel tutorial ("How the monokernel removes launch
overhead": prefill, decode, LM-head sampling in one kernel) assume.  Where the
pages leave a step open the plainest reading is taken:

* RoPE is the "rotate-half" form pairing dims (i, i + hd/2);
  inv_freq_i = fp32(theta ** (-2i/hd)); the angle is the fp32 product
  fp32(pos) * inv_freq_i; cos/sin are taken of that fp32 angle.
* RMSNorm is x / sqrt(mean(x^2) + eps) * g.
* Attention scale is 1/sqrt(hd); GQA query head i reads KV head
  i // (Hq/Hkv); softmax subtracts the row max.
* K and V are stored in the cache as bf16 (round to nearest even) and read
  back exactly; everything else is float64.
* Argmax takes the lowest index among equal maxima.
"""
import numpy as np

F64 = np.float64


# ----------------------------------------------------------------- storage types
def bf16_bits_to_f64(bits):
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(F64)


def fp16_bits_to_f64(bits):
    return np.asarray(bits).view(np.float16).astype(F64)


def round_to_bf16(x):
    """float -> nearest bf16 value (ties to even), returned as float64.

    The value is first rounded to float32 (round to nearest even), then to the
    8-bit significand of bf16 (round to nearest even)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(F64)


# ----------------------------------------------------------------- building blocks
def rmsnorm(x, g, eps):
    """RMSNorm: x * (mean(x^2) + eps)^(-1/2) * g."""
    x = np.asarray(x, F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope_inv_freq(head_dim, theta):
    """inv_freq_i = theta^(-2i/hd), i < hd/2, rounded to float32."""
    i = np.arange(head_dim // 2, dtype=F64)
    return (theta ** (-(2.0 * i) / head_dim)).astype(np.float32)


def rope_cos_sin(pos, head_dim, theta):
    """cos/sin of the float32 angle fp32(pos) * inv_freq_i, as float64."""
    ang = (np.float32(pos) * rope_inv_freq(head_dim, theta)).astype(np.float32)
    a = ang.astype(F64)
    return np.cos(a), np.sin(a)


def rope(v, pos, theta):
    """Rotate-half RoPE of v[..., hd] at position pos."""
    v = np.asarray(v, F64)
    hd = v.shape[-1]
    h = hd // 2
    c, s = rope_cos_sin(pos, hd, theta)
    x1, x2 = v[..., :h], v[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(s):
    s = np.asarray(s, F64)
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_head(q, K, V):
    """One query head over n cached positions: softmax(K q / sqrt(hd)) V."""
    hd = q.shape[-1]
    p = softmax(K @ q / np.sqrt(F64(hd)))
    return p @ V


def gqa_attention(q, K, V):
    """q [Hq, hd]; K, V [Hkv, n, hd]; query head i uses KV head i // (Hq/Hkv)."""
    hq, hkv = q.shape[0], K.shape[0]
    rep = hq // hkv
    return np.stack([attention_head(q[i], K[i // rep], V[i // rep]) for i in range(hq)])


def silu(x):
    x = np.asarray(x, F64)
    return x / (1.0 + np.exp(-x))


def swiglu(gate, up):
    return silu(gate) * up


def argmax_lowest(logits):
    """Index of the maximum; the lowest index wins among equal values."""
    logits = np.asarray(logits)
    if np.isnan(logits).any():
        raise ValueError("NaN logit")
    return int(np.flatnonzero(logits == logits.max())[0])


# ----------------------------------------------------------------- the model
class Model:
    """Float64 weights of one model plus its shape.

    ``weights`` maps names to bf16/fp16 bit arrays (``synthetic.generate_weights``)
    or, for quantised models, to already-dequantised float arrays supplied by
    ``quant``.  ``cache=False`` widens each matrix at use (slow, low memory).
    """

    def __init__(self, shape, weights, base_dtype="bf16", cache=True, dequantised=None):
        self.s = shape
        self.w = weights
        self.base = base_dtype
        self.cache = cache
        self.deq = dequantised or {}
        self._f = {}

    def W(self, name):
        if name in self.deq:
            return self.deq[name]
        if name in self._f:
            return self._f[name]
        bits = self.w[name]
        a = bf16_bits_to_f64(bits) if self.base == "bf16" else fp16_bits_to_f64(bits)
        if self.cache:
            self._f[name] = a
        return a

    def new_cache(self, max_seq):
        s = self.s
        shp = (s.n_layers, s.n_kv_heads, max_seq, s.head_dim)
        return {"K": np.zeros(shp, F64), "V": np.zeros(shp, F64)}


def decode_step(m: Model, kv, tok, pos, want_logits=True):
    """One token through the decoder at position ``pos``; writes KV[pos].

    Returns the logits (float64 [V]) or None when ``want_logits`` is False.
    """
    s = m.s
    x = m.W("embed")[tok].copy()
    for l in range(s.n_layers):
        h = rmsnorm(x, m.W(f"l{l}.attn_norm"), s.rms_eps)
        q = (m.W(f"l{l}.wq") @ h).reshape(s.n_q_heads, s.head_dim)
        k = (m.W(f"l{l}.wk") @ h).reshape(s.n_kv_heads, s.head_dim)
        v = (m.W(f"l{l}.wv") @ h).reshape(s.n_kv_heads, s.head_dim)
        q = rope(q, pos, s.rope_theta)
        k = rope(k, pos, s.rope_theta)
        kv["K"][l, :, pos] = round_to_bf16(k)
        kv["V"][l, :, pos] = round_to_bf16(v)
        o = gqa_attention(q, kv["K"][l, :, : pos + 1], kv["V"][l, :, : pos + 1])
        x = x + m.W(f"l{l}.wo") @ o.reshape(-1)
        h = rmsnorm(x, m.W(f"l{l}.ffn_norm"), s.rms_eps)
        x = x + m.W(f"l{l}.wdown") @ swiglu(m.W(f"l{l}.wgate") @ h, m.W(f"l{l}.wup") @ h)
    if not want_logits:
        return None
    return m.W("lm_head") @ rmsnorm(x, m.W("final_norm"), s.rms_eps)


def prefill(m: Model, kv, prompt):
    """Positions 0..P-2 through the decoder (KV writes only).

    Returns (pending token, its position): the last prompt token is fed by the
    first decode step, which emits the first new token."""
    for p, t in enumerate(prompt[:-1]):
        decode_step(m, kv, int(t), p, want_logits=False)
    return int(prompt[-1]), len(prompt) - 1


def greedy(m: Model, prompt, n_steps, max_seq=None):
    """Greedy decode: returns (ids [n_steps], logits [n_steps, V])."""
    kv = m.new_cache(max_seq or (len(prompt) + n_steps))
    tok, pos = prefill(m, kv, prompt)
    ids, logits = [], []
    for _ in range(n_steps):
        lg = decode_step(m, kv, tok, pos)
        tok = argmax_lowest(lg)
        ids.append(tok)
        logits.append(lg)
        pos += 1
    return np.array(ids, np.int32), np.stack(logits)


def teacher_forced(m: Model, prompt, forced, max_seq=None):
    """Decode with the input of step s fixed to ``forced[s]``.

    Step 0 feeds the last prompt token; step s > 0 feeds forced[s-1] (the
    oracle's own greedy tokens when checking a GPU run).  Returns logits
    [len(forced), V]."""
    n = len(forced)
    kv = m.new_cache(max_seq or (len(prompt) + n))
    tok, pos = prefill(m, kv, prompt)
    out = []
    for s_ in range(n):
        out.append(decode_step(m, kv, tok, pos))
        tok = int(forced[s_])
        pos += 1
    return np.stack(out)


def forward_full(m: Model, tokens, last=None, kv_out=None):
    """All positions at once with a causal mask (matrix form).

    K and V are rounded to bf16 exactly as the cache stores them.  Returns the
    logits for every position [T, V], or for the last ``last`` positions only
    (the final norm and LM head are then applied to those rows alone).  With a
    list ``kv_out``, each layer's cache entries (K, V), float64 arrays
    [Hkv, T, hd] of bf16 values, are appended to it."""
    s = m.s
    T = len(tokens)
    x = m.W("embed")[np.asarray(tokens)].copy()
    rep = s.n_q_heads // s.n_kv_heads
    mask = np.triu(np.full((T, T), -np.inf), 1)
    for l in range(s.n_layers):
        h = rmsnorm(x, m.W(f"l{l}.attn_norm"), s.rms_eps)
        q = (h @ m.W(f"l{l}.wq").T).reshape(T, s.n_q_heads, s.head_dim)
        k = (h @ m.W(f"l{l}.wk").T).reshape(T, s.n_kv_heads, s.head_dim)
        v = (h @ m.W(f"l{l}.wv").T).reshape(T, s.n_kv_heads, s.head_dim)
        q = np.stack([rope(q[p], p, s.rope_theta) for p in range(T)])
        k = round_to_bf16(np.stack([rope(k[p], p, s.rope_theta) for p in range(T)]))
        v = round_to_bf16(v)
        if kv_out is not None:
            kv_out.append((k.transpose(1, 0, 2).copy(), v.transpose(1, 0, 2).copy()))
        o = np.empty((T, s.n_q_heads, s.head_dim))
        for i in range(s.n_q_heads):
            g = i // rep
            sc = q[:, i] @ k[:, g].T / np.sqrt(F64(s.head_dim)) + mask
            o[:, i] = softmax(sc) @ v[:, g]
        x = x + o.reshape(T, -1) @ m.W(f"l{l}.wo").T
        h = rmsnorm(x, m.W(f"l{l}.ffn_norm"), s.rms_eps)
        x = x + swiglu(h @ m.W(f"l{l}.wgate").T, h @ m.W(f"l{l}.wup").T) @ m.W(f"l{l}.wdown").T
    if last is not None:
        x = x[T - last:]
    return rmsnorm(x, m.W("final_norm"), s.rms_eps) @ m.W("lm_head").T
