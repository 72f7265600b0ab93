"""GPU parity: the persistent decode kernel, called through the C ABI, against
the CPU oracle on the same seeded inputs.

Bars (from the decode-path contract): dequantisation bit-exact; token
bookkeeping exact; teacher-forced logits within max|dlogit| <= 1e-2 *
max|logit| per step with >= 99% argmax agreement (fp32 accumulation on the
GPU, float64 oracle).
"""
import numpy as np
import pytest

import synthetic
from oracle import llama as L
from oracle import quant as Q

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


_WEIGHTS = {}


def weights_for(name):
    w = synthetic.get_workload(name)
    key = (w.seed, w.base_dtype, w.n_layers, w.d_model)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        _WEIGHTS[key] = synthetic.generate_weights(w)
    return _WEIGHTS[key]


def oracle_model(w, weights):
    if w.wdtype in ("int8", "int4", "fp8"):
        deq, _ = Q.quantised_model_weights(w, weights, w.wdtype)
        return L.Model(w, weights, w.base_dtype, dequantised=deq)
    return L.Model(w, weights, w.base_dtype)


def check_logits(gpu, ref, tol=TOL, label=""):
    """Per step max|dlogit| <= tol * max|logit_oracle|, >= 99% argmax agreement.
    Prints the worst step's relative error (visible with -s / -rA)."""
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu))
    rel = np.empty(ref.shape[0])
    for s in range(ref.shape[0]):
        err = np.abs(gpu[s] - ref[s]).max()
        scale = np.abs(ref[s]).max()
        rel[s] = err / scale
        assert err <= tol * scale, f"step {s}: max|dlogit| {err:.3e} > {tol} * {scale:.3e}"
    agree = np.mean(gpu.argmax(axis=1) == np.array([L.argmax_lowest(r) for r in ref]))
    print(f"{label} steps={ref.shape[0]} max_rel_err={rel.max():.3e} (step {int(rel.argmax())}) "
          f"median_rel_err={np.median(rel):.3e} argmax_agreement={agree:.4f}")
    assert agree >= 0.99, f"argmax agreement {agree:.3f}"
    return agree


# ------------------------------------------------------------------ dequantisation
QUANTISE = {"int8": (Q.quantize_int8_rows, Q.dequant_int8), "int4": (Q.quantize_int4_g128, Q.dequant_int4),
            "fp8": (Q.quantize_fp8_g128, Q.dequant_fp8)}


@pytest.mark.parametrize("wd", ["int8", "int4", "fp8"])
def test_device_dequant_bit_exact(mk, wd):
    torch = _torch()
    w = synthetic.get_workload("tiny").with_(wdtype=wd)
    weights = weights_for("tiny")
    desc = mk.make_desc(w)
    blob = mk.pack_model(desc, weights)
    dev = torch.from_numpy(blob).cuda()
    for name, tid in mk.GEMV_SOURCES:
        for layer in range(w.n_layers):
            src = synthetic.bits_to_f32(weights[f"l{layer}.{name}"], "bf16")
            q, s = QUANTISE[wd][0](src)
            want = QUANTISE[wd][1](q, s)
            got = mk.debug_dequant(desc, dev, tid, layer, *src.shape).cpu().numpy()
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (name, layer)
    src = synthetic.bits_to_f32(weights["lm_head"], "bf16")
    q, s = QUANTISE[wd][0](src)
    want = QUANTISE[wd][1](q, s)
    got = mk.debug_dequant(desc, dev, mk.MK_T_LM_HEAD, 0, *src.shape).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ------------------------------------------------------------------ tiny model
@pytest.mark.parametrize("sms,chunks", [(0, 0), (7, 3), (1, 1), (152, 5), (0, 64)])
def test_tiny_teacher_forced(mk, sms, chunks):
    # (0, 64): enough partials that per-group merge tasks run (most chunks empty)
    w = synthetic.get_workload("tiny")
    weights = weights_for("tiny")
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights), mk.make_config(sms=sms, attn_chunks=chunks))
    prompt = synthetic.generate_prompt(w)
    om = oracle_model(w, weights)
    ids_o, logits_o = L.greedy(om, prompt, w.decode_steps)
    dec.prefill(prompt)
    forced = np.concatenate([prompt[-1:], ids_o[:-1]]).astype(np.int32)
    lg, ids = dec.teacher_forced(forced)
    check_logits(lg, logits_o)
    # the kernel's own argmax agrees with argmax of the logits it wrote
    assert np.array_equal(ids, lg.argmax(axis=1))
    assert dec.state()[0] == len(prompt) - 1 + w.decode_steps


def test_tiny_greedy_bookkeeping(mk):
    w = synthetic.get_workload("tiny")
    weights = weights_for("tiny")
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights))
    prompt = synthetic.generate_prompt(w)
    ids_o, _ = L.greedy(oracle_model(w, weights), prompt, w.decode_steps)
    dec.prefill(prompt)
    n0 = dec.launch_count()
    ids = dec.decode(w.decode_steps)
    assert dec.launch_count() - n0 == 1          # the whole decode is one launch
    pos, pending = dec.state()
    assert pos == len(prompt) + w.decode_steps - 1 and pending == ids[-1]
    assert ids.shape == (w.decode_steps,)
    # free-running greedy: identical until a near-tie; the tiny model has wide margins
    assert np.array_equal(ids, ids_o)
    # decoding in two calls gives the same stream as one call
    dec.prefill(prompt)
    a = dec.decode(10)
    b = dec.decode(w.decode_steps - 10)
    assert np.array_equal(np.concatenate([a, b]), ids)
    # rewind and replay
    dec.set_state(len(prompt) - 1, int(prompt[-1]))
    assert np.array_equal(dec.decode(w.decode_steps), ids)


def test_tiny_capacity_and_state_errors(mk):
    w = synthetic.get_workload("tiny")
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights_for("tiny")))
    with pytest.raises(mk.MKError) as e:
        dec.decode(1)
    assert e.value.status == mk.MK_ERR_INVALID_ARG  # no prefill yet
    prompt = synthetic.generate_prompt(w)
    dec.prefill(prompt)
    room = w.max_seq - (len(prompt) - 1)   # KV slots pos .. max_seq-1
    with pytest.raises(mk.MKError) as e:
        dec.decode(room + 1)
    assert e.value.status == mk.MK_ERR_CAPACITY
    assert dec.decode(room).shape == (room,)
    with pytest.raises(mk.MKError) as e:
        dec.prefill(np.zeros(w.max_seq + 1, np.int32))
    assert e.value.status == mk.MK_ERR_CAPACITY


def test_prefill_single_token_and_empty_chunks(mk):
    # prompt of one token: no prefill launch; attention at pos 0 over one
    # position with more chunks than positions (empty chunks must merge out)
    w = synthetic.get_workload("tiny")
    weights = weights_for("tiny")
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights), mk.make_config(attn_chunks=4))
    prompt = synthetic.generate_prompt(w)[:1]
    ids_o, logits_o = L.greedy(oracle_model(w, weights), prompt, 6)
    dec.prefill(prompt)
    lg, _ = dec.teacher_forced(np.concatenate([prompt, ids_o[:-1]]).astype(np.int32))
    check_logits(lg, logits_o)


def test_watchdog_returns_timeout(mk):
    torch = _torch()
    import ctypes
    buf = torch.zeros(32, dtype=torch.int32, device="cuda")
    st = mk.load().mk_debug_watchdog(20000, ctypes.c_void_p(buf.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mk.MK_ERR_TIMEOUT
    # the context is still usable
    assert int((buf + 1).sum().item()) == 32 + int(buf.sum().item())


# ------------------------------------------------------------------ full-size models
def _full_size(mk, name, n_forced, sms=0, prompt_len=None, workload=None, cfg=None):
    w = workload or synthetic.get_workload(name)
    weights = synthetic.generate_weights(w) if workload else weights_for(name)
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights), cfg or mk.make_config(sms=sms))
    prompt = synthetic.generate_prompt(w, prompt_len)
    forced_tail = synthetic.gen.random_tokens(w, n_forced - 1, 7)
    dec.prefill(prompt)
    lg, ids = dec.teacher_forced(np.concatenate([prompt[-1:], forced_tail]).astype(np.int32))
    dec.close()
    om = oracle_model(w, weights)
    ref = L.forward_full(om, np.concatenate([prompt, forced_tail]), last=n_forced)
    return lg, ref, ids


@pytest.mark.parametrize("name", ["llama-1b", "llama-1b-int8", "llama-1b-int4", "llama-1b-fp8"])
def test_1b_teacher_forced(mk, name):
    # every step of the bench's timed window: positions 127..382, split-KV
    # chunks growing from ~22 to 64 positions (two tiles and the next-tile prefetch)
    w = synthetic.get_workload(name)
    lg, ref, ids = _full_size(mk, name, w.decode_steps)
    check_logits(lg, ref, label=name)
    assert np.array_equal(ids, lg.argmax(axis=1))


@pytest.mark.parametrize("wd", ["int8", "int4", "fp8"])
@pytest.mark.parametrize("sms", [0, 7])
def test_tiny_quantised_teacher_forced(mk, wd, sms):
    # the fused FFN with quantised codes: one 512-byte line per column block
    w = synthetic.get_workload("tiny").with_(wdtype=wd)
    weights = weights_for("tiny")
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights), mk.make_config(sms=sms))
    ir = mk.mk_build_ir(desc, mk.make_config(sms=sms), dec.launch_info()["ctas"])
    assert "ffn" in {mk.OPS[t["op"]] for t in ir["tasks"]}
    prompt = synthetic.generate_prompt(w)
    om = oracle_model(w, weights)
    ids_o, logits_o = L.greedy(om, prompt, w.decode_steps)
    dec.prefill(prompt)
    lg, ids = dec.teacher_forced(np.concatenate([prompt[-1:], ids_o[:-1]]).astype(np.int32))
    check_logits(lg, logits_o, label=f"tiny-{wd}-sms{sms}")
    assert np.array_equal(ids, lg.argmax(axis=1))
    dec.close()


def _pow2_scaled(bits, k):
    # bf16 bits times 2^k: exact (no value of these weights under- or overflows)
    f = synthetic.bits_to_f32(bits, "bf16") * np.float32(2.0 ** k)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


@pytest.mark.parametrize("wd", ["int8", "int4"])
def test_integer_dot_input_range(mk, wd):
    # int8/int4 GEMVs multiply their codes by a fixed-point copy of the input
    # whose step D = 2^E follows max|x| (c15b).  The ends of that range on the
    # tiny model: all-zero inputs (every other forced token has a zero
    # embedding row, so layer 0's QKV input vanishes and D falls back to 1),
    # attention outputs about 2^-4 of the usual (W_v scaled: O's input takes
    # a smaller E) and SwiGLU outputs about 2^8 of the usual (W_up scaled: the
    # down projection's input takes a larger E).  W_v is not scaled further:
    # the split-KV partials are fp16 values of v's magnitude, and below fp16's
    # normal range (6.1e-5) they lose precision whatever the GEMV does.
    w = synthetic.get_workload("tiny").with_(wdtype=wd)
    weights = dict(weights_for("tiny"))
    for layer in range(w.n_layers):
        weights[f"l{layer}.wv"] = _pow2_scaled(weights[f"l{layer}.wv"], -4)
        weights[f"l{layer}.wup"] = _pow2_scaled(weights[f"l{layer}.wup"], 8)
    prompt = synthetic.generate_prompt(w)
    forced_tail = synthetic.gen.random_tokens(w, w.decode_steps - 1, 11)
    emb = weights["embed"].copy()
    emb[np.unique(forced_tail[::2])] = 0
    weights["embed"] = emb
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights))
    dec.prefill(prompt)
    lg, ids = dec.teacher_forced(np.concatenate([prompt[-1:], forced_tail]).astype(np.int32))
    ref = L.forward_full(oracle_model(w, weights), np.concatenate([prompt, forced_tail]), last=w.decode_steps)
    check_logits(lg, ref, label=f"tiny-{wd}-input-range")
    assert np.array_equal(ids, lg.argmax(axis=1))
    dec.close()


@pytest.mark.parametrize("wd", ["int8", "int4", "fp8"])
def test_8b_shape_quantised_teacher_forced(mk, wd):
    # d_model 4096: 16 lines per column block, i.e. a block spans 2 (int8) or
    # 4 (int4) ring batches; the int4 group scales change every 4 blocks
    w = synthetic.get_workload("llama3-8b-8k").with_(n_layers=2, prompt_len=96, decode_steps=128, wdtype=wd,
                                                     vocab=32000)
    lg, ref, ids = _full_size(mk, w.name, w.decode_steps, workload=w)
    check_logits(lg, ref, label=f"8b-shape-2L-{wd}")
    assert np.array_equal(ids, lg.argmax(axis=1))


def test_2b_fp16_teacher_forced(mk):
    # fp16 weights, head_dim 128, d_model 2560: GEMV rows split over two warps,
    # the fused FFN with 10 lines per column block, merge tasks (16 chunks);
    # the config's 512-token prompt and 64 decode steps
    lg, ref, ids = _full_size(mk, "llama-2b-fp16", 64)
    check_logits(lg, ref, label="llama-2b-fp16")
    assert np.array_equal(ids, lg.argmax(axis=1))


def test_8b_shape_teacher_forced(mk):
    # Llama-3-8B widths (d 4096, F 14336, vocab 128256, theta 5e5, head_dim 128)
    # at two layers and a 96-token prompt: 16-line column blocks, two-warp rows,
    # the 17-bit argmax index; one split-KV chunk per head (no merge tasks);
    # 128 steps, so that the 99% argmax gate allows one near-tie flip
    w = synthetic.get_workload("llama3-8b-8k").with_(n_layers=2, prompt_len=96, decode_steps=128)
    lg, ref, ids = _full_size(mk, w.name, w.decode_steps, workload=w)
    check_logits(lg, ref, label="8b-shape-2L-96")
    assert np.array_equal(ids, lg.argmax(axis=1))


def test_8b_shape_8k_context(mk):
    # The benchmarked long-context path: the 8B widths at two layers with the
    # config's real 8,192-token prompt, at the default launch shape, so each KV
    # head is split into many chunks of hundreds of positions (over ten
    # attention tiles each), the fp16 partials are merged by merge tasks, and
    # 100 teacher-forced steps follow.  The vocabulary is cut to 32000 to keep the
    # float64 oracle's LM head small (the 17-bit index is covered above).
    w = synthetic.get_workload("llama3-8b-8k").with_(n_layers=2, vocab=32000, decode_steps=100)
    desc = mk.make_desc(w)
    torch = _torch()
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    ir = mk.mk_build_ir(desc, mk.make_config(), n_sms)
    ops = [mk.OPS[t["op"]] for t in ir["tasks"]]
    chunks = ops.count("attn") // (w.n_layers * w.n_kv_heads)
    assert "merge" in ops and chunks > 8, (chunks, set(ops))
    assert (w.prompt_len + w.decode_steps) / chunks > 10 * 32  # chunks span more than ten 32-position tiles
    lg, ref, ids = _full_size(mk, w.name, w.decode_steps, workload=w)
    check_logits(lg, ref, label=f"8b-shape-2L-8k C={chunks}")
    assert np.array_equal(ids, lg.argmax(axis=1))


# ------------------------------------------------------------------ argmax ties
def _lm_row_ranges(mk, desc, n_sms):
    """Row range [r0, r1) and CTA of every LM-head task of the lowering."""
    ir = mk.mk_build_ir(desc, mk.make_config(), n_sms)
    out = []
    for t in ir["tasks"]:
        if mk.OPS[t["op"]] == "lm":
            lo, hi = next((a[2], a[3]) for a in t["acc"] if a[1] == mk.MK_ACC_WRITE and a[4] != 0)
            out.append((lo // 4, hi // 4, t["sm"]))
    return sorted(out)


@pytest.mark.parametrize("where", ["other_cta", "same_batch"])
def test_argmax_ties_take_the_lowest_index(mk, where):
    """Two LM-head rows hold the same bf16 values, scaled up so that they are
    often the maximum; their logits must be bit-identical and the kernel must
    return the lower index, both teacher-forced and in a greedy run.  The pair
    sits on two different CTAs (the cross-CTA atomicMax key) or in one warp
    batch (the in-warp reduction)."""
    torch = _torch()
    w = synthetic.get_workload("tiny")
    weights = dict(weights_for("tiny"))
    desc = mk.make_desc(w)
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    rr = _lm_row_ranges(mk, desc, n_sms)
    if where == "other_cta":
        a, b = rr[1], rr[-2]
        assert a[2] != b[2]
        j1, j2 = a[0], b[1] - 1
    else:
        a = next(r for r in rr if r[1] - r[0] >= 2)
        j1, j2 = a[0], a[0] + 1  # rows 0 and 1 of the task: one batch of warp group 0
    lm = weights["lm_head"].copy()
    row = synthetic.bits_to_f32(lm[3], "bf16") * np.float32(20.0)
    lm[j1] = lm[j2] = synthetic.gen._f32_to_bf16_bits(row)
    weights["lm_head"] = lm
    dec = mk.Decoder(desc, mk.pack_model(desc, weights))
    prompt = synthetic.generate_prompt(w)
    om = oracle_model(w, weights)
    ids_o, logits_o = L.greedy(om, prompt, w.decode_steps)
    dec.prefill(prompt)
    forced = np.concatenate([prompt[-1:], ids_o[:-1]]).astype(np.int32)
    lg, ids = dec.teacher_forced(forced)
    check_logits(lg, logits_o, label=f"tie {where} ({j1}, {j2})")
    assert np.array_equal(lg[:, j1].view(np.uint32), lg[:, j2].view(np.uint32))
    want = np.array([L.argmax_lowest(r) for r in lg])
    assert np.array_equal(ids, want)
    wins = int(np.sum(ids == j1))
    assert wins >= 3 and not np.any(ids == j2), (wins, ids)
    # greedy: one launch whose every step reads the key the previous step wrote
    dec.set_state(len(prompt) - 1, int(prompt[-1]))
    g = dec.decode(w.decode_steps)
    assert np.array_equal(g, ids_o) and not np.any(g == j2)
    dec.close()


# ------------------------------------------------------------------ several handles
def test_two_handles_share_one_kernel(mk):
    """The 1B and tiny models run the same kernel instantiation (bf16, head_dim
    64) with different shared-memory sizes.  Creating the tiny handle after the
    1B one must not stop the 1B handle's launches, nor the static entry point's."""
    torch = _torch()
    w1, wt = synthetic.get_workload("llama-1b"), synthetic.get_workload("tiny")
    d1, dt = mk.make_desc(w1), mk.make_desc(wt)
    wts1 = weights_for("llama-1b")
    big = mk.Decoder(d1, mk.pack_model(d1, wts1))
    wtt = synthetic.generate_weights(wt)
    small = mk.Decoder(dt, mk.pack_model(dt, wtt))
    assert big.launch_info()["smem_bytes"] > small.launch_info()["smem_bytes"]
    p1, pt = synthetic.generate_prompt(w1), synthetic.generate_prompt(wt)
    # 1B, teacher-forced against the oracle, after the tiny handle exists
    big.prefill(p1)
    tail = synthetic.gen.random_tokens(w1, 3, 7)
    lg, _ = big.teacher_forced(np.concatenate([p1[-1:], tail]).astype(np.int32))
    check_logits(lg, L.forward_full(oracle_model(w1, wts1), np.concatenate([p1, tail]), last=4), label="1b+tiny")
    # tiny, greedy against the oracle
    small.prefill(pt)
    ids_small = small.decode(4)
    assert np.array_equal(ids_small, L.greedy(oracle_model(wt, wtt), pt, 4)[0])
    # both again, then the static entry point with each model
    big.set_state(len(p1) - 1, int(p1[-1]))
    ids_big = big.decode(4)
    assert np.all((ids_big >= 0) & (ids_big < w1.vocab))
    for dec, desc, prompt, ids in ((big, d1, p1, ids_big), (small, dt, pt, ids_small)):
        got = mk.decode_static(desc, dec.weights, dec.kv, len(prompt) - 1, int(prompt[-1]), 4)
        assert np.array_equal(got, ids)
    small.set_state(len(pt) - 1, int(pt[-1]))
    assert np.array_equal(small.decode(4), ids_small)
    torch.cuda.synchronize()
    big.close()
    small.close()


# ------------------------------------------------------------------ run-to-run spread
def test_repeated_launch_spread(mk):
    """The fused FFN ends with red.add from every CTA into the residual, in an
    order that changes from run to run, so repeated launches on the same input
    differ in the last bits.  Bound that spread far below the parity gate."""
    w = synthetic.get_workload("llama-1b")
    weights = weights_for("llama-1b")
    desc = mk.make_desc(w)
    dec = mk.Decoder(desc, mk.pack_model(desc, weights))
    prompt = synthetic.generate_prompt(w)
    forced = np.concatenate([prompt[-1:], synthetic.gen.random_tokens(w, 31, 7)]).astype(np.int32)
    runs = []
    for _ in range(4):
        dec.prefill(prompt)
        runs.append(dec.teacher_forced(forced)[0])
    dec.close()
    spread = max(float((np.abs(r - runs[0]).max(axis=1) / np.abs(runs[0]).max(axis=1)).max()) for r in runs[1:])
    print(f"run-to-run max|dlogit|/max|logit| over 4 launches x 32 steps: {spread:.3e}")
    assert spread <= 1e-3


def test_schedule_grid_search_on_tiny(mk, capsys, tmp_path):
    # the tuner validates, checks against the oracle's teacher-forced logits and
    # times each grid point
    from decode_megakernel_02_gb300 import tune
    import json
    w = synthetic.get_workload("tiny")
    weights = weights_for("tiny")
    prompt, forced = tune.forced_stream(w, 8)
    ref = L.forward_full(oracle_model(w, weights), np.concatenate([prompt, forced[1:]]), last=8)
    np.save(tmp_path / "ref.npy", ref.astype(np.float32))
    tune.main(["--workload", "tiny", "--chunks", "0,2,4", "--sms", "0,7", "--reps", "1",
               "--token-select", "0,1", "--reference", str(tmp_path / "ref.npy")])
    out = json.loads(capsys.readouterr().out)
    assert out["agreement_reference"] == "reference file"
    assert len(out["points"]) == 12
    assert all(p["status"] == "ok" for p in out["points"]), out["points"]
    assert all(p["tokens_per_s"] > 0 for p in out["points"])
    # a reference that no configuration matches rejects every point
    np.save(tmp_path / "bad.npy", (ref + 0.05 * np.abs(ref).max()).astype(np.float32))
    tune.main(["--workload", "tiny", "--chunks", "0", "--reps", "1", "--reference", str(tmp_path / "bad.npy")])
    out = json.loads(capsys.readouterr().out)
    assert [p["status"] for p in out["points"]] == ["rejected: logits differ from the reference file"]
