"""GPU parity of the tensor-core chunked prefill (mk_schedule_config.prefill_chunk):
the bf16 KV cache it leaves equals the oracle's cache entries within 1e-2 of
each layer's largest entry, and the decode steps that follow pass the
teacher-forced logit gate (max|dlogit| <= 1e-2 * max|logit|, >= 99% argmax
agreement).  The prompt GEMMs take 16-bit activations (the operand type of
the tensor cores), so the cache is not bit-equal to the float64 oracle's;
its error is about one bf16 rounding of the values."""
import time

import numpy as np
import pytest

import synthetic
from oracle import llama as L

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def mk():
    _torch()
    from decode_megakernel_02_gb300 import build
    build.build()
    import decode_megakernel_02_gb300 as m
    m.load()
    return m


def _kv(dec, w):
    """The handle's cache as float32 [L][2][Hkv][max_seq][hd]."""
    torch = _torch()
    return dec.kv.view(torch.bfloat16).float().reshape(w.n_layers, 2, w.n_kv_heads, w.max_seq, w.head_dim).cpu().numpy()


def _run(mk, w, chunk, n_forced, weights=None):
    weights = weights or synthetic.generate_weights(w)
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights), mk.make_config(prefill_chunk=chunk))
    prompt = synthetic.generate_prompt(w)
    torch = _torch()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dec.prefill(prompt)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3
    kv = _kv(dec, w)
    tail = synthetic.gen.random_tokens(w, n_forced - 1, 7)
    lg, ids = dec.teacher_forced(np.concatenate([prompt[-1:], tail]).astype(np.int32))
    dec.close()
    om = L.Model(w, weights, w.base_dtype)
    kv_o = []
    ref = L.forward_full(om, np.concatenate([prompt, tail]), last=n_forced, kv_out=kv_o)
    P = len(prompt) - 1  # positions the prefill wrote
    worst = 0.0
    for l, (k, v) in enumerate(kv_o):
        for j, want in ((0, k), (1, v)):
            got = kv[l, j, :, :P]
            err = np.abs(got - want[:, :P]).max()
            scale = np.abs(want[:, :P]).max()
            worst = max(worst, err / scale)
            assert err <= TOL * scale, (l, j, err, scale)
    for s in range(n_forced):
        err = np.abs(lg[s] - ref[s]).max()
        assert err <= TOL * np.abs(ref[s]).max(), (s, err)
    agree = np.mean(lg.argmax(1) == np.array([L.argmax_lowest(r) for r in ref]))
    print(f"{w.name} chunk={chunk}: prefill of {P} positions {ms:.1f} ms, KV worst {worst:.2e} of the largest entry, "
          f"{n_forced} decode steps, argmax agreement {agree:.3f}")
    assert agree >= 0.99 or n_forced < 100 and agree >= 1 - 1.0 / n_forced
    return ms


@pytest.mark.parametrize("prompt,chunk", [(8, 128), (300, 128), (129, 128)])
def test_tiny_prefill(mk, prompt, chunk):
    # one ragged chunk; three chunks (chunk boundaries inside the prompt);
    # a prompt of exactly one full chunk of positions
    w = synthetic.get_workload("tiny").with_(prompt_len=prompt)
    _run(mk, w, chunk, 16)


def test_1b_prefill(mk):
    w = synthetic.get_workload("llama-1b")
    _run(mk, w, 128, 32)


def test_2b_fp16_prefill(mk):
    # fp16 operands (kind::f16 with fp16 A and B), head_dim 128, five query
    # heads per KV head, a 512-token prompt in two chunks
    w = synthetic.get_workload("llama-2b-fp16")
    _run(mk, w, 256, 16)


def test_8b_shape_8k_prefill(mk):
    """The 8B widths at two layers with the real 8,192-token prompt in chunks
    of 1024: column-block down projection (3-D tensor map), 16-line blocks,
    attention of later chunks over the cache of earlier ones."""
    w = synthetic.get_workload("llama3-8b-8k").with_(n_layers=2, vocab=32000, decode_steps=100)
    ms = _run(mk, w, 1024, 100)
    assert ms > 0


def test_prefill_chunk_errors(mk):
    w = synthetic.get_workload("tiny")
    with pytest.raises(mk.MKError) as e:  # not a multiple of 128
        mk.Decoder(mk.make_desc(w), mk.pack_model(mk.make_desc(w), synthetic.generate_weights(w)),
                   mk.make_config(prefill_chunk=100))
    assert e.value.status == mk.MK_ERR_INVALID_ARG
    wq = w.with_(wdtype="int8")
    with pytest.raises(mk.MKError) as e:  # the prompt GEMMs need 16-bit weights
        mk.Decoder(mk.make_desc(wq), mk.pack_model(mk.make_desc(wq), synthetic.generate_weights(wq)),
                   mk.make_config(prefill_chunk=128))
    assert e.value.status == mk.MK_ERR_UNSUPPORTED
