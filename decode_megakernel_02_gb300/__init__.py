"""Python binding of libmk (the batch-1 decode megakernel C ABI).

Argument marshalling only: every step of decode runs in the library's CUDA
kernel.  PyTorch is used for device memory and streams.  The functions keep
the C names (``mk_create``, ``mk_prefill``, ``mk_decode`` ...); ``Decoder``
bundles the caller-owned buffers of one model.  There is no CPU fallback:
loading fails loudly when ``libmk.so`` has not been built.
"""
import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmk.so")

# ------------------------------------------------------------------ constants (include/mk.h)
MK_OK, MK_ERR_INVALID_ARG, MK_ERR_UNSUPPORTED, MK_ERR_SCHEDULE_INVALID = 0, 1, 2, 3
MK_ERR_CAPACITY, MK_ERR_CUDA, MK_ERR_TIMEOUT, MK_ERR_DEVICE = 4, 5, 6, 7
MK_W_BF16, MK_W_FP16, MK_W_INT8_ROW, MK_W_INT4_G128, MK_W_FP8_E4M3 = 0, 1, 2, 3, 4
MK_FLAG_PROJ_BIAS, MK_FLAG_TIED_HEAD, MK_FLAG_ROPE_SCALING = 1, 2, 4
(MK_T_EMBED, MK_T_LM_HEAD, MK_T_FINAL_NORM, MK_T_ATTN_NORM, MK_T_FFN_NORM, MK_T_WQ, MK_T_WK, MK_T_WV,
 MK_T_WO, MK_T_WGATE, MK_T_WUP, MK_T_WDOWN) = range(12)
MK_ACC_READ, MK_ACC_WRITE, MK_ACC_ATOMIC = 1, 2, 3
MK_BUF_OUTPUT = 1
MK_IR_MAX_WAITS = 2
MK_STATIC_SCRATCH_BYTES = 8 << 20
OPS = {1: "qkv", 2: "attn", 3: "o", 4: "gu", 5: "down", 6: "lm", 7: "fin", 8: "ffn", 9: "merge", 10: "select"}
MK_MAX_TOP_K = 64
WDTYPES = {"bf16": MK_W_BF16, "fp16": MK_W_FP16, "int8": MK_W_INT8_ROW, "int4": MK_W_INT4_G128,
           "fp8": MK_W_FP8_E4M3}
STATUS_NAMES = {0: "MK_OK", 1: "MK_ERR_INVALID_ARG", 2: "MK_ERR_UNSUPPORTED", 3: "MK_ERR_SCHEDULE_INVALID",
                4: "MK_ERR_CAPACITY", 5: "MK_ERR_CUDA", 6: "MK_ERR_TIMEOUT", 7: "MK_ERR_DEVICE"}
THREADS_PER_CTA = 256  # eight warps


class mk_model_desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("d_ffn", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("max_seq", ctypes.c_int32), ("wdtype", ctypes.c_int32), ("base_dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class mk_schedule_config(ctypes.Structure):
    _fields_ = [("sms", ctypes.c_int32), ("rows_in_flight", ctypes.c_int32), ("attn_chunks", ctypes.c_int32),
                ("watchdog_ms", ctypes.c_int32), ("token_select", ctypes.c_int32),
                ("prefill_chunk", ctypes.c_int32)]


class mk_sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("seed", ctypes.c_uint64),
                ("eos_id", ctypes.c_int32)]


class mk_ir_task(ctypes.Structure):
    _fields_ = [("sm", ctypes.c_int32), ("op", ctypes.c_int32), ("layer", ctypes.c_int32),
                ("n_waits", ctypes.c_int32), ("wait_ctr", ctypes.c_int32 * MK_IR_MAX_WAITS),
                ("wait_count", ctypes.c_int32 * MK_IR_MAX_WAITS),
                ("wait_epoch_off", ctypes.c_int32 * MK_IR_MAX_WAITS), ("signal_ctr", ctypes.c_int32),
                ("acc_begin", ctypes.c_int32), ("n_acc", ctypes.c_int32)]


class mk_ir_access(ctypes.Structure):
    _fields_ = [("buf", ctypes.c_int32), ("kind", ctypes.c_int32), ("lo", ctypes.c_int64),
                ("hi", ctypes.c_int64), ("stride", ctypes.c_int64), ("grow", ctypes.c_int64)]


class mk_ir(ctypes.Structure):
    _fields_ = [("n_sms", ctypes.c_int32), ("n_tasks", ctypes.c_int32), ("n_counters", ctypes.c_int32),
                ("n_buffers", ctypes.c_int32), ("n_acc", ctypes.c_int32),
                ("tasks", ctypes.POINTER(mk_ir_task)), ("acc", ctypes.POINTER(mk_ir_access)),
                ("queue", ctypes.POINTER(ctypes.c_int32)), ("queue_off", ctypes.POINTER(ctypes.c_int32)),
                ("buf_flags", ctypes.POINTER(ctypes.c_int32)), ("ctr_buf", ctypes.POINTER(ctypes.c_int32))]


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_DESC = ctypes.POINTER(mk_model_desc)
_CFG = ctypes.POINTER(mk_schedule_config)

# name -> (restype, argtypes); the full set include/mk.h declares
SIGNATURES = {
    "mk_packed_size": (_I32, [_DESC, ctypes.POINTER(_SZ)]),
    "mk_pack_tensor": (_I32, [_DESC, _I32, _I32, _P, _P, _SZ]),
    "mk_tensor_layout": (_I32, [_DESC, _I32, _I32, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ),
                                ctypes.POINTER(_I32), ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "mk_quantize_int8": (_I32, [_P, _I64, _I64, _P, _P]),
    "mk_quantize_int4": (_I32, [_P, _I64, _I64, _P, _P]),
    "mk_quantize_fp8": (_I32, [_P, _I64, _I64, _P, _P]),
    "mk_kv_cache_size": (_I32, [_DESC, ctypes.POINTER(_SZ)]),
    "mk_workspace_size": (_I32, [_DESC, _CFG, _I32, ctypes.POINTER(_SZ)]),
    "mk_build_ir": (_I32, [_DESC, _CFG, _I32, ctypes.POINTER(ctypes.POINTER(mk_ir))]),
    "mk_free_ir": (None, [ctypes.POINTER(mk_ir)]),
    "mk_validate_ir": (_I32, [ctypes.POINTER(mk_ir), ctypes.c_char_p, _SZ]),
    "mk_validate_schedule": (_I32, [_DESC, _CFG, _I32, ctypes.c_char_p, _SZ]),
    "mk_create": (_I32, [_DESC, _CFG, _P, _SZ, _P, _SZ, _P, _SZ, _P, ctypes.POINTER(_P)]),
    "mk_prefill": (_I32, [_P, _P, _I32]),
    "mk_decode": (_I32, [_P, _I32, _P]),
    "mk_decode_async": (_I32, [_P, _I32, _P, _P, _P]),
    "mk_finish": (_I32, [_P]),
    "mk_get_state": (_I32, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "mk_set_state": (_I32, [_P, _I32, _I32]),
    "mk_get_launch_info": (_I32, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32), ctypes.POINTER(_I32),
                                  ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "mk_launch_count": (_I64, [_P]),
    "mk_set_sampling": (_I32, [_P, ctypes.POINTER(mk_sampling)]),
    "mk_last_steps": (_I32, [_P]),
    "mk_last_error": (ctypes.c_char_p, [_P]),
    "mk_destroy": (None, [_P]),
    "mk_decode_static": (_I32, [_DESC, _CFG, _P, _SZ, _P, _SZ, _I32, _I32, _I32, _P, _P, _P]),
    "mk_debug_dequant": (_I32, [_DESC, _P, _I32, _I32, _P, _P]),
    "mk_debug_set_trace": (_I32, [_P, _P, _I32]),
    "mk_debug_watchdog": (_I32, [_I32, _P, _P]),
}

_lib = None


def load(path=LIB_PATH):
    """Load libmk.so (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with decode_megakernel_02_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MKError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(st, handle=None):
    if st != MK_OK:
        msg = load().mk_last_error(handle)
        raise MKError(st, msg.decode() if msg else "")
    return st


# ------------------------------------------------------------------ descriptors
def make_desc(workload, max_seq=None, wdtype=None, flags=0):
    """mk_model_desc for a synthetic.Workload-like object."""
    wd = WDTYPES[wdtype or workload.wdtype]
    base = WDTYPES[workload.base_dtype]
    return mk_model_desc(workload.n_layers, workload.d_model, workload.n_q_heads, workload.n_kv_heads,
                         workload.head_dim, workload.d_ffn, workload.vocab, workload.rms_eps,
                         workload.rope_theta, max_seq or workload.max_seq, wd, base, flags)


def make_config(sms=0, rows_in_flight=0, attn_chunks=0, watchdog_ms=0, token_select=0, prefill_chunk=0):
    return mk_schedule_config(sms, rows_in_flight, attn_chunks, watchdog_ms, token_select, prefill_chunk)


# ------------------------------------------------------------------ host calls
def mk_packed_size(desc):
    n = _SZ()
    _check(load().mk_packed_size(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def mk_kv_cache_size(desc):
    n = _SZ()
    _check(load().mk_kv_cache_size(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def mk_workspace_size(desc, cfg=None, n_sms=0):
    n = _SZ()
    _check(load().mk_workspace_size(ctypes.byref(desc), ctypes.byref(cfg) if cfg else None, n_sms,
                                    ctypes.byref(n)))
    return n.value


def mk_pack_tensor(desc, tensor, layer, src, blob):
    src = np.ascontiguousarray(src, dtype=np.uint16)
    assert blob.dtype == np.uint8 and blob.flags.c_contiguous
    _check(load().mk_pack_tensor(ctypes.byref(desc), tensor, layer, src.ctypes.data, blob.ctypes.data, blob.nbytes))


def mk_tensor_layout(desc, tensor, layer=0):
    off, stride = _SZ(), _SZ()
    first, step, rows = _I32(), _I32(), _I32()
    _check(load().mk_tensor_layout(ctypes.byref(desc), tensor, layer, ctypes.byref(off), ctypes.byref(stride),
                                   ctypes.byref(first), ctypes.byref(step), ctypes.byref(rows)))
    return dict(offset=off.value, stride=stride.value, first_row=first.value, row_step=step.value,
                rows=rows.value)


def mk_quantize_int8(w):
    w = np.ascontiguousarray(w, np.float32)
    n, k = w.shape
    q = np.empty((n, k), np.int8)
    s = np.empty(n, np.uint16)
    _check(load().mk_quantize_int8(w.ctypes.data, n, k, q.ctypes.data, s.ctypes.data))
    return q, s.view(np.float16)


def mk_quantize_int4(w):
    w = np.ascontiguousarray(w, np.float32)
    n, k = w.shape
    q = np.empty((n, k), np.int8)
    s = np.empty((n, k // 128), np.uint16)
    _check(load().mk_quantize_int4(w.ctypes.data, n, k, q.ctypes.data, s.ctypes.data))
    return q, s.view(np.float16)


def mk_quantize_fp8(w):
    w = np.ascontiguousarray(w, np.float32)
    n, k = w.shape
    q = np.empty((n, k), np.uint8)
    s = np.empty((n, k // 128), np.uint16)
    _check(load().mk_quantize_fp8(w.ctypes.data, n, k, q.ctypes.data, s.ctypes.data))
    return q, s.view(np.float16)


def mk_validate_schedule(desc, cfg=None, n_sms=152):
    why = ctypes.create_string_buffer(1024)
    st = load().mk_validate_schedule(ctypes.byref(desc), ctypes.byref(cfg) if cfg else None, n_sms, why, 1024)
    return st, why.value.decode()


# ------------------------------------------------------------------ schedule IR
def mk_build_ir(desc, cfg=None, n_sms=152):
    """Lower desc/cfg and return the IR as plain Python data (see oracle.schedule_sim)."""
    p = ctypes.POINTER(mk_ir)()
    _check(load().mk_build_ir(ctypes.byref(desc), ctypes.byref(cfg) if cfg else None, n_sms, ctypes.byref(p)))
    try:
        return ir_to_dict(p.contents)
    finally:
        load().mk_free_ir(p)


def ir_to_dict(ir):
    tasks = []
    for i in range(ir.n_tasks):
        t = ir.tasks[i]
        acc = []
        for a in range(t.acc_begin, t.acc_begin + t.n_acc):
            x = ir.acc[a]
            acc.append((x.buf, x.kind, x.lo, x.hi, x.stride, x.grow))
        tasks.append({"sm": t.sm, "op": t.op, "layer": t.layer,
                      "waits": [(t.wait_ctr[w], t.wait_count[w], t.wait_epoch_off[w]) for w in range(t.n_waits)],
                      "signal": t.signal_ctr, "acc": acc})
    queues = [[ir.queue[j] for j in range(ir.queue_off[s], ir.queue_off[s + 1])] for s in range(ir.n_sms)]
    outputs = [b for b in range(ir.n_buffers) if ir.buf_flags[b] & MK_BUF_OUTPUT]
    tagged = {c: ir.ctr_buf[c] for c in range(ir.n_counters) if ir.ctr_buf and ir.ctr_buf[c] >= 0}
    return {"n_sms": ir.n_sms, "n_counters": ir.n_counters, "n_buffers": ir.n_buffers, "outputs": outputs,
            "tasks": tasks, "queues": queues, "tagged": tagged}


def mk_validate_ir(irdict):
    """Run the library's validator on a (possibly mutated) IR dict: (status, why)."""
    T = len(irdict["tasks"])
    accs = [a for t in irdict["tasks"] for a in t["acc"]]
    tasks = (mk_ir_task * max(1, T))()
    acc = (mk_ir_access * max(1, len(accs)))()
    k = 0
    for i, t in enumerate(irdict["tasks"]):
        x = tasks[i]
        x.sm, x.op, x.layer = t["sm"], t.get("op", 0), t.get("layer", 0)
        x.n_waits = len(t["waits"])
        for w, (c, cnt, off) in enumerate(t["waits"][:MK_IR_MAX_WAITS]):
            x.wait_ctr[w], x.wait_count[w], x.wait_epoch_off[w] = c, cnt, off
        if len(t["waits"]) > MK_IR_MAX_WAITS:
            x.n_waits = len(t["waits"])
        x.signal_ctr = t["signal"]
        x.acc_begin, x.n_acc = k, len(t["acc"])
        for a in t["acc"]:
            acc[k].buf, acc[k].kind, acc[k].lo, acc[k].hi, acc[k].stride, acc[k].grow = a
            k += 1
    flat = [j for q in irdict["queues"] for j in q]
    queue = (_I32 * max(1, len(flat)))(*flat)
    offs = [0]
    for q in irdict["queues"]:
        offs.append(offs[-1] + len(q))
    queue_off = (_I32 * len(offs))(*offs)
    nb = irdict["n_buffers"]
    flags = (_I32 * max(1, nb))(*[MK_BUF_OUTPUT if b in irdict.get("outputs", []) else 0 for b in range(nb)])
    nc = irdict["n_counters"]
    tagged = irdict.get("tagged", {})
    ctr_buf = (_I32 * max(1, nc))(*[tagged.get(c, -1) for c in range(nc)])
    ir = mk_ir(irdict["n_sms"], T, nc, nb, len(accs), tasks, acc, queue, queue_off, flags, ctr_buf)
    why = ctypes.create_string_buffer(1024)
    st = load().mk_validate_ir(ctypes.byref(ir), why, 1024)
    return st, why.value.decode()


# ------------------------------------------------------------------ packing helpers
GEMV_SOURCES = (("wq", MK_T_WQ), ("wk", MK_T_WK), ("wv", MK_T_WV), ("wo", MK_T_WO), ("wgate", MK_T_WGATE),
                ("wup", MK_T_WUP), ("wdown", MK_T_WDOWN))


def pack_model(desc, weights):
    """Pack a dict of bf16/fp16 bit arrays (synthetic.generate_weights layout)
    into one host blob (numpy uint8) with the library's packer."""
    blob = np.zeros(mk_packed_size(desc), np.uint8)
    mk_pack_tensor(desc, MK_T_EMBED, 0, weights["embed"], blob)
    mk_pack_tensor(desc, MK_T_LM_HEAD, 0, weights["lm_head"], blob)
    mk_pack_tensor(desc, MK_T_FINAL_NORM, 0, weights["final_norm"], blob)
    for l in range(desc.n_layers):
        mk_pack_tensor(desc, MK_T_ATTN_NORM, l, weights[f"l{l}.attn_norm"], blob)
        mk_pack_tensor(desc, MK_T_FFN_NORM, l, weights[f"l{l}.ffn_norm"], blob)
        for name, tid in GEMV_SOURCES:
            mk_pack_tensor(desc, tid, l, weights[f"l{l}.{name}"], blob)
    return blob


# ------------------------------------------------------------------ device runtime
class Decoder:
    """One model on the current CUDA device: packed weights, KV cache and
    workspace are torch-allocated device buffers owned here; ``mk_create``
    validates the schedule before anything is launched."""

    def __init__(self, desc, blob, cfg=None, stream=None, device="cuda"):
        import torch
        self.torch = torch
        self.desc = desc
        self.cfg = cfg or make_config()
        lib = load()
        self.stream = stream or torch.cuda.current_stream()
        self.weights = torch.empty(len(blob), dtype=torch.uint8, device=device)
        self.weights.copy_(torch.from_numpy(blob))
        self.kv = torch.zeros(mk_kv_cache_size(desc), dtype=torch.uint8, device=device)
        self.ws = torch.zeros(mk_workspace_size(desc, self.cfg), dtype=torch.uint8, device=device)
        torch.cuda.synchronize()
        h = _P()
        _check(lib.mk_create(ctypes.byref(desc), ctypes.byref(self.cfg), self.weights.data_ptr(),
                             self.weights.numel(), self.kv.data_ptr(), self.kv.numel(), self.ws.data_ptr(),
                             self.ws.numel(), _P(self.stream.cuda_stream), ctypes.byref(h)))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            load().mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, tokens):
        t = np.ascontiguousarray(tokens, np.int32)
        _check(load().mk_prefill(self.h, t.ctypes.data, len(t)), self.h)

    def decode(self, n_steps, out=None):
        """Greedy decode (synchronous); returns int32 ids (numpy)."""
        if out is None:
            out = np.empty(n_steps, np.int32)
        elif not (isinstance(out, np.ndarray) and out.dtype == np.int32 and out.flags.c_contiguous
                  and out.size >= n_steps):
            raise ValueError("out must be a C-contiguous int32 numpy array of at least n_steps elements")
        _check(load().mk_decode(self.h, n_steps, out.ctypes.data), self.h)
        return out

    def decode_async(self, n_steps, forced=None, out_ids=None, logits=None):
        """Enqueue one launch; tensors are device tensors (or None)."""
        torch = self.torch
        for t, dt, n, name in ((forced, torch.int32, n_steps, "forced"), (out_ids, torch.int32, n_steps, "out_ids"),
                               (logits, torch.float32, n_steps * self.desc.vocab, "logits")):
            if t is not None and not (t.device == self.weights.device and t.dtype == dt and t.is_contiguous()
                                      and t.numel() >= n):
                raise ValueError(f"{name} must be a contiguous {dt} tensor on {self.weights.device} "
                                 f"with at least {n} elements")
        ptr = (lambda t: t.data_ptr() if t is not None else None)
        _check(load().mk_decode_async(self.h, n_steps, ptr(forced), ptr(out_ids), ptr(logits)), self.h)

    def finish(self):
        _check(load().mk_finish(self.h), self.h)

    def state(self):
        pos, pending = _I32(), _I32()
        _check(load().mk_get_state(self.h, ctypes.byref(pos), ctypes.byref(pending)), self.h)
        return pos.value, pending.value

    def set_state(self, pos, pending):
        _check(load().mk_set_state(self.h, pos, pending), self.h)

    def launch_info(self):
        v = [_I32() for _ in range(5)]
        _check(load().mk_get_launch_info(self.h, *[ctypes.byref(x) for x in v]), self.h)
        return dict(zip(("ctas", "threads", "smem_bytes", "rows_in_flight", "n_tasks"), [x.value for x in v]))

    def set_trace(self, buf=None, records_per_cta=0):
        """Per-task timestamps of later launches into a device uint64 tensor
        [ctas, records_per_cta, 8] (None disables)."""
        _check(load().mk_debug_set_trace(self.h, buf.data_ptr() if buf is not None else None,
                                         records_per_cta), self.h)

    def launch_count(self):
        return load().mk_launch_count(self.h)

    def set_sampling(self, temperature=0.0, top_k=0, seed=0, eos_id=-1):
        """Token selection of later launches (mk_set_sampling): greedy at
        temperature 0, else Gumbel-max sampling over all tokens or the top_k
        logits; decoding stops after emitting eos_id (-1: never)."""
        s = mk_sampling(float(temperature), int(top_k), int(seed) & 0xFFFFFFFFFFFFFFFF, int(eos_id))
        _check(load().mk_set_sampling(self.h, ctypes.byref(s)), self.h)

    def last_steps(self):
        """Steps the last launch ran (fewer than asked after an EOS stop)."""
        return load().mk_last_steps(self.h)

    def teacher_forced(self, forced_tokens):
        """Feed forced_tokens[s] at step s; returns (logits [n, V] float32, argmax ids [n])."""
        torch = self.torch
        n = len(forced_tokens)
        f = torch.tensor(np.asarray(forced_tokens, np.int32), device=self.weights.device)
        lg = torch.empty((n, self.desc.vocab), dtype=torch.float32, device=self.weights.device)
        ids = torch.empty(n, dtype=torch.int32, device=self.weights.device)
        self.decode_async(n, forced=f, out_ids=ids, logits=lg)
        self.finish()
        return lg.cpu().numpy(), ids.cpu().numpy()


def decode_static(desc, weights, kv, pos, token, n_steps, cfg=None, logits=None, stream=None, out=None):
    """``mk_decode_static``: greedy decode from (pos, token) into the caller's
    KV cache with the library's static device scratch (no allocation on the
    device).  weights/kv/logits are caller-owned device tensors; returns the
    int32 ids (numpy, host)."""
    import torch
    if out is None:
        out = np.empty(n_steps, np.int32)
    elif not (isinstance(out, np.ndarray) and out.dtype == np.int32 and out.flags.c_contiguous
              and out.size >= n_steps):
        raise ValueError("out must be a C-contiguous int32 numpy array of at least n_steps elements")
    if logits is not None and not (logits.is_cuda and logits.dtype == torch.float32 and logits.is_contiguous()
                                   and logits.device == weights.device
                                   and logits.numel() >= n_steps * desc.vocab):
        raise ValueError("logits must be a contiguous float32 tensor on the weights' device with at least "
                         "n_steps * vocab elements")
    st = stream or torch.cuda.current_stream()
    _check(load().mk_decode_static(ctypes.byref(desc), ctypes.byref(cfg) if cfg else None, weights.data_ptr(),
                                   weights.numel() * weights.element_size(), kv.data_ptr(),
                                   kv.numel() * kv.element_size(), pos, token, n_steps, out.ctypes.data,
                                   logits.data_ptr() if logits is not None else None, _P(st.cuda_stream)))
    return out


def debug_dequant(desc, weights_dev, tensor, layer, rows, cols, stream=None):
    """Device dequantisation of one packed tensor (test support)."""
    import torch
    out = torch.empty((rows, cols), dtype=torch.float32, device=weights_dev.device)
    st = stream or torch.cuda.current_stream()
    _check(load().mk_debug_dequant(ctypes.byref(desc), weights_dev.data_ptr(), tensor, layer, out.data_ptr(),
                                   _P(st.cuda_stream)))
    return out
