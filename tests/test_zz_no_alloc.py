"""mk_decode_static (greedy decode with the library's static device scratch,
no device allocation) against the handle path (mk_create + mk_decode_async)
on the same packed weights, prompt and KV state: two calls in a row, ids
identical, logits within the parity tolerance, KV caches alike.

The file name sorts last so that the suite also runs it after every other
GPU test in the same process."""
import gc

import numpy as np
import pytest

import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-2  # max|dlogit| <= TOL * max|logit|, as in the oracle parity tests


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


def _compare(mk, name, steps, cfg):
    torch = _torch()
    w = synthetic.get_workload(name)
    weights = synthetic.generate_weights(w)
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights), cfg)
    prompt = synthetic.generate_prompt(w)
    dec.prefill(prompt)
    kv_static = dec.kv.clone()  # KV of positions 0..len(prompt)-2, before any decode step
    dev = dec.weights.device

    ref_ids, ref_lg = [], []
    for n in steps:  # the existing entry point, two calls in a row
        ids = torch.empty(n, dtype=torch.int32, device=dev)
        lg = torch.empty((n, w.vocab), dtype=torch.float32, device=dev)
        dec.decode_async(n, out_ids=ids, logits=lg)
        dec.finish()
        ref_ids.append(ids.cpu().numpy())
        ref_lg.append(lg.cpu().numpy())

    # every buffer of the static calls exists before the first one
    lgs = [torch.full((n, w.vocab), float("nan"), dtype=torch.float32, device=dev) for n in steps]
    outs = [np.full(n, -1, np.int32) for n in steps]
    gc.collect()  # tensors of earlier tests are freed now, not during the calls below
    torch.cuda.synchronize()
    pos, tok = len(prompt) - 1, int(prompt[-1])
    for i, n in enumerate(steps):
        alloc0 = torch.cuda.memory_allocated()
        free0 = torch.cuda.mem_get_info()[0]
        mk.decode_static(desc, dec.weights, kv_static, pos, tok, n, cfg=cfg, logits=lgs[i], out=outs[i])
        if i > 0:  # after the first call's set-up the device's free memory does not shrink
            assert torch.cuda.mem_get_info()[0] >= free0
        assert torch.cuda.memory_allocated() <= alloc0  # nothing allocated through torch
        pos, tok = pos + n, int(outs[i][-1])

    for i in range(len(steps)):
        got = lgs[i].cpu().numpy()
        assert np.all(np.isfinite(got))
        for s in range(steps[i]):
            err = np.abs(got[s] - ref_lg[i][s]).max()
            assert err <= TOL * np.abs(ref_lg[i][s]).max(), (i, s, err)
        assert np.array_equal(outs[i], ref_ids[i]), (i, outs[i], ref_ids[i])
    a = kv_static.view(torch.bfloat16).float()
    b = dec.kv.view(torch.bfloat16).float()
    assert torch.allclose(a, b, rtol=TOL, atol=TOL * float(b.abs().max()))
    dec.close()


@pytest.mark.parametrize("sms,chunks", [(0, 0), (7, 3)])
def test_static_matches_handle_tiny(mk, sms, chunks):
    _compare(mk, "tiny", (9, 14), mk.make_config(sms=sms, attn_chunks=chunks))


def test_static_matches_handle_1b(mk):
    _compare(mk, "llama-1b", (4, 5), mk.make_config())


def test_static_rejects_oversized_scratch(mk):
    torch = _torch()
    w = synthetic.get_workload("tiny")
    small = mk.make_desc(w)
    big = mk.make_desc(w, max_seq=1 << 20)  # token-id arrays alone exceed the static scratch
    assert mk.mk_workspace_size(big) > mk.MK_STATIC_SCRATCH_BYTES
    dec = mk.Decoder(small, mk.pack_model(small, synthetic.generate_weights(w)))
    with pytest.raises(mk.MKError) as e:
        mk.decode_static(big, dec.weights, dec.kv, 0, 1, 1)
    assert e.value.status == mk.MK_ERR_CAPACITY
    assert "static scratch" in str(e.value)
    # the device is still usable and a fitting model still runs
    prompt = synthetic.generate_prompt(w)
    dec.prefill(prompt)
    ids = mk.decode_static(small, dec.weights, dec.kv, len(prompt) - 1, int(prompt[-1]), 3)
    assert ids.shape == (3,) and np.all((ids >= 0) & (ids < w.vocab))
    torch.cuda.synchronize()
    dec.close()
