"""Host-side checks of the C ABI (no GPU): the library loads and exports every
function include/mk.h declares; the packer and its quantisers produce the
oracle's bytes; the static validator accepts every real lowering and never
accepts a schedule the brute-force simulator finds unsafe."""
import ctypes
import os
import random
import re

import numpy as np
import pytest

import synthetic
from oracle import quant as Q
from oracle import schedule_sim as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mk():
    from decode_megakernel_02_gb300 import build
    build.build()
    import decode_megakernel_02_gb300 as m
    m.load()
    return m


# ------------------------------------------------------------------ exports
def declared_functions():
    text = open(os.path.join(ROOT, "include", "mk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:mk_status|int64_t|int32_t|const char\s*\*|void)\s*\*?\s*(mk_\w+)\s*\(",
                                 text, flags=re.M)))


def test_library_exports_every_declared_function(mk):
    names = declared_functions()
    assert len(names) >= 25
    lib = ctypes.CDLL(os.path.join(ROOT, "decode_megakernel_02_gb300", "libmk.so"))
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding declares a signature for every exported entry point
    assert set(names) == set(mk.SIGNATURES), set(names) ^ set(mk.SIGNATURES)


def test_errors_without_a_device(mk):
    # contract violations are reported before any CUDA call
    w = synthetic.get_workload("tiny")
    d = mk.make_desc(w, flags=mk.MK_FLAG_TIED_HEAD)
    with pytest.raises(mk.MKError) as e:
        mk.mk_packed_size(d)
    assert e.value.status == mk.MK_ERR_UNSUPPORTED
    d = mk.make_desc(w)
    d.head_dim = 96
    with pytest.raises(mk.MKError) as e:
        mk.mk_packed_size(d)
    assert e.value.status == mk.MK_ERR_UNSUPPORTED


def test_int4_row_length_limit(mk):
    # int4 rows carry one fp16 scale per 128 codes in a 128-byte slot trailer,
    # so they are limited to 8192 codes: an unfused FFN (d_model 2560 is not a
    # fused shape for quantised codes) with d_ffn 8320 would need longer down
    # rows.  The fused shapes and rows up to the limit are accepted.
    w = synthetic.get_workload("tiny")
    d = mk.make_desc(w.with_(wdtype="int4", d_model=2560, n_q_heads=20, n_kv_heads=4, d_ffn=8320))
    with pytest.raises(mk.MKError) as e:
        mk.mk_packed_size(d)
    assert e.value.status == mk.MK_ERR_UNSUPPORTED
    assert "int4 rows" in str(e.value)
    assert mk.mk_packed_size(mk.make_desc(w.with_(wdtype="int4", d_model=2560, n_q_heads=20, n_kv_heads=4,
                                                  d_ffn=8192))) > 0
    assert mk.mk_packed_size(mk.make_desc(w.with_(wdtype="int4", d_model=4096, n_q_heads=32, n_kv_heads=8,
                                                  d_ffn=14336))) > 0  # fused: the long rows are columns
    assert mk.mk_packed_size(mk.make_desc(w.with_(wdtype="int8", d_model=2560, n_q_heads=20, n_kv_heads=4,
                                                  d_ffn=8320))) > 0


# ------------------------------------------------------------------ packer
def test_quantisers_match_oracle_bytes(mk):
    rng = np.random.default_rng(5)
    w = synthetic.bits_to_f32(
        (rng.standard_normal((37, 256), np.float32) * 0.02).astype(np.float32).view(np.uint32) >> 16, "bf16")
    w[3] = 0.0  # an all-zero row: scale 0, codes 0
    q, s = mk.mk_quantize_int8(w)
    qo, so = Q.quantize_int8_rows(w)
    assert np.array_equal(q, qo) and np.array_equal(s.view(np.uint16), so.view(np.uint16))
    q, s = mk.mk_quantize_int4(w)
    qo, so = Q.quantize_int4_g128(w)
    assert np.array_equal(q, qo) and np.array_equal(s.view(np.uint16), so.view(np.uint16))
    # FP8 E4M3: the C++ round-to-nearest-even from the format definition and the
    # oracle's nearest-value search agree byte for byte, ties and clamping included
    q, s = mk.mk_quantize_fp8(w)
    qo, so = Q.quantize_fp8_g128(w)
    assert np.array_equal(q, qo) and np.array_equal(s.view(np.uint16), so.view(np.uint16))
    wide = (rng.standard_normal((8, 256)) * 50).astype(np.float32)  # many scales, ties by chance
    assert np.array_equal(mk.mk_quantize_fp8(wide)[0], Q.quantize_fp8_g128(wide)[0])


@pytest.mark.parametrize("wd", ["int8", "int4", "fp8"])
def test_packed_quantised_rows_match_oracle(mk, wd):
    w = synthetic.get_workload("tiny").with_(wdtype=wd)
    weights = synthetic.generate_weights(w)
    desc = mk.make_desc(w)
    blob = mk.pack_model(desc, weights)
    for name, tid in (("wq", mk.MK_T_WQ), ("wup", mk.MK_T_WUP), ("wdown", mk.MK_T_WDOWN)):
        src = synthetic.bits_to_f32(weights[f"l1.{name}"], "bf16")
        lay = mk.mk_tensor_layout(desc, tid, 1)
        K = src.shape[1]
        if lay["stride"] == 0:  # the fused FFN's down projection: column blocks, then the scales
            assert name == "wdown"
            n, BU = src.shape[0], 32 if wd == "int4" else 16
            if wd == "int8":
                q, s = Q.quantize_int8_rows(src)
                codes = q.view(np.uint8).reshape(n, K // BU, 16)
                scales = s.view(np.uint8)
            elif wd == "fp8":
                q, s = Q.quantize_fp8_g128(src)
                codes = q.reshape(n, K // BU, 16)
                scales = np.ascontiguousarray(s.T).view(np.uint8).reshape(-1)
            else:
                q, s = Q.quantize_int4_g128(src)
                codes = Q.pack_int4_nibbles(q).reshape(n, K // BU, 16)
                scales = np.ascontiguousarray(s.T).view(np.uint8).reshape(-1)
            nb = n * K * 16 // BU
            region = blob[lay["offset"]:lay["offset"] + nb].reshape(K // BU, n, 16)
            assert np.array_equal(region, codes.transpose(1, 0, 2)), (wd, name)
            assert np.array_equal(blob[lay["offset"] + nb:lay["offset"] + nb + scales.size], scales.reshape(-1))
            continue
        for r in (0, 1, src.shape[0] - 1):
            row = blob[lay["offset"] + (lay["first_row"] + r * lay["row_step"]) * lay["stride"]:][:lay["stride"]]
            if wd == "int8":
                q, s = Q.quantize_int8_rows(src[r:r + 1])
                want = np.concatenate([q.view(np.uint8)[0], s.view(np.uint8)])
            elif wd == "fp8":
                q, s = Q.quantize_fp8_g128(src[r:r + 1])
                want = np.concatenate([q[0], s.view(np.uint8)[0]])
            else:
                q, s = Q.quantize_int4_g128(src[r:r + 1])
                want = np.concatenate([Q.pack_int4_nibbles(q)[0], s.view(np.uint8)[0]])
            assert np.array_equal(row[:len(want)], want), (name, r)
            assert not row[len(want):].any()
        assert lay["stride"] % 16 == 0 and K > 0


def test_packed_down_column_blocks(mk):
    w = synthetic.get_workload("tiny")
    weights = synthetic.generate_weights(w)
    desc = mk.make_desc(w)
    blob = mk.pack_model(desc, weights)
    lay = mk.mk_tensor_layout(desc, mk.MK_T_WDOWN, 0)
    assert lay["stride"] == 0  # 16-bit weights with the fused FFN: column blocks of 8
    down = np.asarray(weights["l0.wdown"], np.uint16)  # [d][F]
    d, F = down.shape
    region = blob[lay["offset"]:lay["offset"] + d * F * 2].view(np.uint16).reshape(F // 8, d, 8)
    assert np.array_equal(region, down.reshape(d, F // 8, 8).transpose(1, 0, 2))


# ------------------------------------------------------------------ validator
@pytest.mark.parametrize("name,sms,chunks", [("tiny", 152, 0), ("tiny", 7, 3), ("tiny", 1, 1), ("tiny", 2, 4),
                                             ("tiny", 152, 64),
                                             ("llama-1b", 152, 0), ("llama-1b-int8", 152, 0),
                                             ("llama-1b-int4", 64, 2), ("llama-1b-fp8", 152, 0),
                                             ("llama-2b-fp16", 152, 0)])
def test_validator_accepts_real_lowerings(mk, name, sms, chunks):
    w = synthetic.get_workload(name)
    st, why = mk.mk_validate_schedule(mk.make_desc(w), mk.make_config(sms=sms, attn_chunks=chunks), sms)
    assert st == mk.MK_OK, why


@pytest.mark.parametrize("name,sms", [("tiny", 152), ("tiny", 3), ("llama-1b", 152), ("llama3-8b-8k", 152)])
def test_validator_accepts_token_select_lowerings(mk, name, sms):
    """The token-select schedule (an OP_SELECT task after the LM head, the next
    step's first layer waiting on its counter) passes the validator."""
    w = synthetic.get_workload(name)
    cfg = mk.make_config(sms=sms, token_select=1)
    st, why = mk.mk_validate_schedule(mk.make_desc(w), cfg, sms)
    assert st == mk.MK_OK, why
    ir = mk.mk_build_ir(mk.make_desc(w), cfg, sms)
    assert [mk.OPS[t["op"]] for t in ir["tasks"]].count("select") == 1


def test_header_constants_match_the_binding(mk):
    text = open(os.path.join(ROOT, "include", "mk.h")).read()
    m = re.search(r"#define MK_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == mk.MK_STATIC_SCRATCH_BYTES
    assert int(re.search(r"#define MK_MAX_TOP_K (\d+)", text).group(1)) == mk.MK_MAX_TOP_K


def _small_ir(mk, sms, chunks, wdtype=None):
    w = synthetic.get_workload("tiny").with_(n_layers=1)
    if wdtype:
        w = w.with_(wdtype=wdtype)
    return mk.mk_build_ir(mk.make_desc(w, max_seq=16), mk.make_config(sms=sms, attn_chunks=chunks), sms)


def _mutants(ir, rng, n):
    """Structural mutations of a real schedule (thresholds, waits, epoch offsets,
    queue order, task placement, signals, accesses, outputs)."""
    import copy
    out = []
    T = len(ir["tasks"])
    for _ in range(n):
        m = copy.deepcopy(ir)
        kind = rng.randrange(9)
        t = m["tasks"][rng.randrange(T)]
        if kind == 0 and t["waits"]:
            c, k, o = t["waits"][0]
            t["waits"][0] = (c, k + rng.choice([1, 2]), o)
        elif kind == 1 and t["waits"]:
            c, k, o = t["waits"][0]
            t["waits"][0] = (c, max(1, k - 1), o)
        elif kind == 2 and t["waits"]:
            t["waits"].pop(rng.randrange(len(t["waits"])))
        elif kind == 3 and t["waits"]:
            c, k, o = t["waits"][0]
            t["waits"][0] = (c, k, -1 - o)
        elif kind == 4:
            q = m["queues"][rng.randrange(len(m["queues"]))]
            if len(q) >= 2:
                i = rng.randrange(len(q) - 1)
                q[i], q[i + 1] = q[i + 1], q[i]
        elif kind == 5 and len(m["queues"]) > 1:
            s0 = rng.randrange(len(m["queues"]))
            s1 = (s0 + 1) % len(m["queues"])
            if m["queues"][s0]:
                j = m["queues"][s0].pop(rng.randrange(len(m["queues"][s0])))
                m["queues"][s1].insert(rng.randrange(len(m["queues"][s1]) + 1), j)
                m["tasks"][j]["sm"] = s1
        elif kind == 6 and t["signal"] >= 0:
            t["signal"] = rng.randrange(m["n_counters"])
        elif kind == 7 and t["acc"]:
            b, k, lo, hi, st, gr = t["acc"][rng.randrange(len(t["acc"]))]
            t["acc"].append((b, S.WRITE, lo, hi, st, gr))
        elif kind == 8:
            m["outputs"] = []
        out.append(m)
    return out


def _delete_task(m, j):
    """Remove task j from the schedule and renumber the later ones."""
    m["tasks"].pop(j)
    m["queues"] = [[i - (i > j) for i in q if i != j] for q in m["queues"]]


def _more_mutants(ir, rng, n):
    """The kinds of _mutants plus edits of what tasks touch: a dropped access, a
    shrunken or shifted byte range, a deleted task, an access moved to another
    buffer, and a hole in the coverage of a tagged buffer."""
    import copy
    out = []
    base = _mutants(ir, rng, n // 2)
    out.extend(base)
    T = len(ir["tasks"])
    tagged_bufs = set(ir.get("tagged", {}).values())
    for _ in range(n - len(base)):
        m = copy.deepcopy(ir)
        kind = rng.randrange(5)
        j = rng.randrange(T)
        t = m["tasks"][j]
        if kind == 0 and t["acc"]:
            t["acc"].pop(rng.randrange(len(t["acc"])))
        elif kind == 1 and t["acc"]:
            i = rng.randrange(len(t["acc"]))
            b, k, lo, hi, st, gr = t["acc"][i]
            d = rng.choice([4, 8, 16, 64, max(4, (hi - lo) // 2)])
            how = rng.randrange(3)
            if how == 0:
                lo = min(hi, lo + d)          # shrink from below
            elif how == 1:
                hi = max(lo, hi - d)          # shrink from above
            else:
                lo, hi = lo + d, hi + d       # shift
            t["acc"][i] = (b, k, lo, hi, st, gr)
        elif kind == 2:
            _delete_task(m, j)
        elif kind == 3 and t["acc"]:
            i = rng.randrange(len(t["acc"]))
            b, k, lo, hi, st, gr = t["acc"][i]
            t["acc"][i] = (rng.choice([x for x in range(m["n_buffers"]) if x != b]), k, lo, hi, st, gr)
        elif kind == 4 and tagged_bufs:
            writers = [(jj, i) for jj, tt in enumerate(m["tasks"]) for i, x in enumerate(tt["acc"])
                       if x[0] in tagged_bufs and x[1] != S.READ]
            jj, i = rng.choice(writers)
            b, k, lo, hi, st, gr = m["tasks"][jj]["acc"][i]
            d = rng.choice([8, 16, max(8, (hi - lo) // 2)])
            m["tasks"][jj]["acc"][i] = (b, k, lo, max(lo, hi - d), st, gr) if rng.randrange(2) else \
                (b, k, min(hi, lo + d), hi, st, gr)
        out.append(m)
    return out


# (sms, chunks, weight type, layers, mutants): 1- and 2-layer tiny schedules,
# all with tagged q/k/v counters; about 5,400 mutants in all
CORPUS = [(2, 1, None, 1, 1500), (3, 2, None, 1, 1500), (2, 1, "int8", 1, 800), (3, 2, None, 2, 1000),
          (2, 2, "int4", 2, 600)]


def test_validator_mutation_corpus(mk):
    """AutoMegaKernel explainer ("Main contributions"): the validator rejects
    every unsafe schedule of an adversarial corpus (no false accept) and
    accepts every real lowering.  Ground truth is the brute-force simulator."""
    totals = dict(mutants=0, unsafe=0, rejected=0, false_accepts=0, safe_rejected=0)
    examples = []
    for sms, chunks, wd, layers, n in CORPUS:
        w = synthetic.get_workload("tiny").with_(n_layers=layers)
        if wd:
            w = w.with_(wdtype=wd)
        ir = mk.mk_build_ir(mk.make_desc(w, max_seq=16), mk.make_config(sms=sms, attn_chunks=chunks), sms)
        assert ir["tagged"], "the corpus starts from schedules with tagged counters"
        assert S.verdict(ir)[0] and mk.mk_validate_ir(ir)[0] == mk.MK_OK
        rng = random.Random(7919 * sms + 31 * chunks + layers)
        for m in _more_mutants(ir, rng, n):
            safe, why = S.verdict(m)
            st, vwhy = mk.mk_validate_ir(m)
            totals["mutants"] += 1
            totals["unsafe"] += not safe
            totals["rejected"] += st != mk.MK_OK
            if st == mk.MK_OK and not safe:
                totals["false_accepts"] += 1
                examples.append(why)
            totals["safe_rejected"] += safe and st != mk.MK_OK
    print("validator corpus:", totals)
    assert totals["mutants"] >= 5000
    assert totals["false_accepts"] == 0, examples[:3]
    assert totals["unsafe"] >= 1000  # the corpus is adversarial


@pytest.mark.parametrize("sms,chunks,wd,n", [(2, 1, None, 60), (3, 2, None, 60), (2, 1, "int8", 60),
                                             (2, 64, None, 12)])
def test_validator_never_accepts_what_the_simulator_rejects(mk, sms, chunks, wd, n):
    ir = _small_ir(mk, sms, chunks, wd)
    assert S.verdict(ir)[0], S.verdict(ir)[1]
    assert mk.mk_validate_ir(ir)[0] == mk.MK_OK
    rng = random.Random(1000 * sms + chunks)
    false_accepts, rejected = [], 0
    for m in _mutants(ir, rng, n):
        safe, why = S.verdict(m)
        st, vwhy = mk.mk_validate_ir(m)
        if st == mk.MK_OK and not safe:
            false_accepts.append(why)
        rejected += st != mk.MK_OK
    assert not false_accepts, false_accepts[:3]
    assert rejected > n // 6  # the corpus does exercise the validator


def test_tuner_agreement_rule():
    from decode_megakernel_02_gb300 import tune
    rng = np.random.default_rng(3)
    ref = rng.standard_normal((5, 64))
    assert tune.agrees(ref.copy(), ref)
    near = ref + 0.5e-2 * np.abs(ref).max(axis=1, keepdims=True) * rng.uniform(-1, 1, ref.shape)
    assert tune.agrees(near, ref) == bool(np.mean(near.argmax(1) == ref.argmax(1)) >= 0.99)
    far = ref.copy()
    far[2, 7] += 0.02 * np.abs(ref[2]).max()
    assert not tune.agrees(far, ref)
    bad = ref.copy()
    bad[0, 0] = np.nan
    assert not tune.agrees(bad, ref)


# ------------------------------------------------------------------ tagged counters
def _tagged_case(mk):
    """A small real schedule whose q/k/v counter is tagged, one attention task
    waiting on it, and a QKV producer whose rows that task reads."""
    ir = _small_ir(mk, 3, 2)
    assert ir["tagged"], "the lowering tags the q/k/v counter"
    c, b = next(iter(ir["tagged"].items()))
    a = next(i for i, t in enumerate(ir["tasks"]) if any(w[0] == c for w in t["waits"]))
    reads = [x for x in ir["tasks"][a]["acc"] if x[0] == b]
    q = next(i for i, t in enumerate(ir["tasks"]) if t["signal"] == c and any(
        y[0] == b and y[1] != S.READ and y[2] < x[3] and x[2] < y[3] for y in t["acc"] for x in reads))
    return ir, c, b, a, q


def test_tagged_wait_orders_only_its_buffer(mk):
    ir, c, b, a, q = _tagged_case(mk)
    assert mk.mk_validate_ir(ir)[0] == mk.MK_OK
    # a side channel: the producer also writes bytes of another buffer that the waiter reads
    other = 3  # the hidden-state buffer, unused by this fused schedule
    ir["tasks"][q]["acc"].append((other, S.WRITE, 0, 8, 0, 0))
    ir["tasks"][a]["acc"].append((other, S.READ, 0, 8, 0, 0))
    st, why = mk.mk_validate_ir(ir)
    assert st != mk.MK_OK and "race" in why, why
    # through a counter word the same access is ordered
    ir["tagged"] = {}
    st, why = mk.mk_validate_ir(ir)
    assert st == mk.MK_OK, why


def test_tagged_wait_must_be_covered_and_current(mk):
    ir, c, b, a, q = _tagged_case(mk)
    import copy
    m = copy.deepcopy(ir)
    m["tasks"][q]["acc"] = [y for y in m["tasks"][q]["acc"] if y[0] != b]  # the producer stops writing its rows
    st, why = mk.mk_validate_ir(m)
    assert st != mk.MK_OK and "tagged wait" in why, why
    assert not S.verdict(m)[0]
    m = copy.deepcopy(ir)
    m["tasks"][a]["waits"] = [(w[0], w[1], -1) if w[0] == c else w for w in m["tasks"][a]["waits"]]
    st, why = mk.mk_validate_ir(m)
    assert st != mk.MK_OK and "tagged wait" in why, why
    assert not S.verdict(m)[0]


@pytest.mark.parametrize("name", ["llama-1b", "llama-2b-fp16", "llama3-8b-8k"])
def test_lowering_tags_every_layer(mk, name):
    """The QKV -> attention hop of every layer travels as tagged values at the
    bench's launch shape, and the validator accepts the result."""
    w = synthetic.get_workload(name)
    ir = mk.mk_build_ir(mk.make_desc(w), mk.make_config(), 152)
    assert len(ir["tagged"]) == w.n_layers
    assert set(ir["tagged"].values()) == {1}  # the q/k/v buffer
    waiters = [t for t in ir["tasks"] if any(c in ir["tagged"] for c, _, _ in t["waits"])]
    assert waiters and {mk.OPS[t["op"]] for t in waiters} == {"attn"}
    assert mk.mk_validate_ir(ir)[0] == mk.MK_OK
