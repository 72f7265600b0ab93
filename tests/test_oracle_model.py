"""Whole-model pins for the oracle (CPU only)."""
import math

import numpy as np
import pytest
import torch

import synthetic
from oracle import llama as L

rng = np.random.default_rng(99)


def _bf16(x):
    """bf16 rounding by torch's own conversion (round to nearest even)."""
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _rms(x, eps):
    return [xi / math.sqrt(sum(v * v for v in x) / len(x) + eps) for xi in x]


def _matvec(W, x):
    return [sum(W[r][k] * x[k] for k in range(len(x))) for r in range(len(W))]


def _tiny_shape(n_layers=1):
    return synthetic.get_workload("tiny").with_(
        n_layers=n_layers, d_model=8, n_q_heads=4, n_kv_heads=2, head_dim=4, d_ffn=6, vocab=10,
        prompt_len=5, decode_steps=3)


def _float_model(shape, overrides):
    w = {}
    d, qd, kd, f, v = shape.d_model, shape.q_dim, shape.kv_dim, shape.d_ffn, shape.vocab
    shp = {"wq": (qd, d), "wk": (kd, d), "wv": (kd, d), "wo": (d, qd),
           "wgate": (f, d), "wup": (f, d), "wdown": (d, f)}
    w["embed"] = rng.standard_normal((v, d))
    w["lm_head"] = rng.standard_normal((v, d))
    w["final_norm"] = np.ones(d)
    for l in range(shape.n_layers):
        for t, s in shp.items():
            w[f"l{l}.{t}"] = rng.standard_normal(s) * 0.3
        w[f"l{l}.attn_norm"] = np.ones(d)
        w[f"l{l}.ffn_norm"] = np.ones(d)
    w.update(overrides(shape))
    return L.Model(shape, {}, dequantised=w), w


def test_zero_keys_attention_is_running_mean_of_values():
    shape = _tiny_shape()
    m, w = _float_model(shape, lambda s: {"l0.wk": np.zeros((s.kv_dim, s.d_model)),
                                          "l0.wgate": np.zeros((s.d_ffn, s.d_model))})
    prompt = np.array([3, 7, 1, 9, 4], np.int32)
    logits = L.teacher_forced(m, prompt, [0])[0]
    eps, hd, rep = shape.rms_eps, shape.head_dim, shape.n_q_heads // shape.n_kv_heads
    vs = []
    for t in prompt:
        h = _rms(list(w["embed"][t]), eps)
        vs.append(_bf16(_matvec(w["l0.wv"], h)))
    o = []
    for i in range(shape.n_q_heads):
        g = i // rep
        for d_ in range(hd):
            o.append(sum(v[g * hd + d_] for v in vs) / len(vs))
    x = [a + b for a, b in zip(w["embed"][prompt[-1]], _matvec(w["l0.wo"], o))]
    want = _matvec(w["lm_head"], _rms(x, eps))
    assert np.allclose(logits, want, rtol=1e-12, atol=1e-12)


def test_ffn_only_path_closed_form():
    shape = _tiny_shape()
    m, w = _float_model(shape, lambda s: {"l0.wo": np.zeros((s.d_model, s.q_dim))})
    prompt = np.array([2, 8], np.int32)
    logits = L.teacher_forced(m, prompt, [0])[0]
    eps = shape.rms_eps
    e = list(w["embed"][8])
    h = _rms(e, eps)
    gt, up = _matvec(w["l0.wgate"], h), _matvec(w["l0.wup"], h)
    act = [g / (1 + math.exp(-g)) * u for g, u in zip(gt, up)]
    x = [a + b for a, b in zip(e, _matvec(w["l0.wdown"], act))]
    assert np.allclose(logits, _matvec(w["lm_head"], _rms(x, eps)), rtol=1e-12, atol=1e-12)


def test_identity_layer_passes_residual_through():
    s2 = _tiny_shape(2)
    m2, w2 = _float_model(s2, lambda s: {"l1.wo": np.zeros((s.d_model, s.q_dim)),
                                         "l1.wdown": np.zeros((s.d_model, s.d_ffn))})
    s1 = _tiny_shape(1)
    w1 = {k: v for k, v in w2.items() if not k.startswith("l1.")}
    m1 = L.Model(s1, {}, dequantised=w1)
    prompt = np.array([1, 2, 3, 4], np.int32)
    assert np.allclose(L.teacher_forced(m2, prompt, [5, 6]), L.teacher_forced(m1, prompt, [5, 6]), rtol=1e-13)


def test_incremental_decode_equals_full_causal_recompute():
    shape = synthetic.get_workload("tiny")
    m = L.Model(shape, synthetic.generate_weights(shape))
    prompt = synthetic.generate_prompt(shape)
    forced = synthetic.gen.random_tokens(shape, 6, 0)
    inc = L.teacher_forced(m, prompt, forced)
    seq = np.concatenate([prompt, forced[:-1]])
    full = L.forward_full(m, seq)[len(prompt) - 1:]
    scale = np.abs(full).max()
    assert np.abs(inc - full).max() <= 1e-9 * scale


def test_greedy_bookkeeping():
    shape = synthetic.get_workload("tiny")
    m = L.Model(shape, synthetic.generate_weights(shape))
    prompt = synthetic.generate_prompt(shape)
    ids, logits = L.greedy(m, prompt, 4)
    assert ids.shape == (4,) and logits.shape == (4, shape.vocab)
    for s in range(4):
        assert ids[s] == int(np.argmax(logits[s]))
    # teacher forcing on the greedy tokens reproduces the greedy logits exactly
    assert np.array_equal(L.teacher_forced(m, prompt, ids), logits)


def test_forward_full_kv_equals_incremental_cache():
    """The cache entries forward_full reports are the ones incremental decode
    writes (same bf16 rounding, same positions)."""
    w = synthetic.get_workload("tiny").with_(n_layers=2)
    m = L.Model(w, synthetic.generate_weights(w))
    toks = synthetic.generate_prompt(w, 9)
    kv_full = []
    L.forward_full(m, toks, kv_out=kv_full)
    cache = m.new_cache(len(toks))
    for p, t in enumerate(toks):
        L.decode_step(m, cache, int(t), p, want_logits=False)
    for l, (k, v) in enumerate(kv_full):
        assert np.allclose(k, cache["K"][l], rtol=0, atol=1e-12 + 8e-3 * np.abs(k).max())
        assert np.allclose(v, cache["V"][l], rtol=0, atol=1e-12 + 8e-3 * np.abs(v).max())
