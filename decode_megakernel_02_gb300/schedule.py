"""Schedule tool: explain, validate and serialise a lowered decode schedule.

Netra Kernel summary, "Section details": the engine compiles a deterministic
artifact (no timestamps) and its CLI explains and statically validates a
compiled schedule.  This tool does the same for this library's lowering,
host only, through the C ABI (mk_build_ir, mk_validate_ir):

    python -m decode_megakernel_02_gb300.schedule explain  --workload llama-1b
    python -m decode_megakernel_02_gb300.schedule validate --workload llama3-8b-8k
    python -m decode_megakernel_02_gb300.schedule dump     --workload tiny --out tiny.json
    python -m decode_megakernel_02_gb300.schedule validate --ir tiny.json

`dump` writes the IR as canonical JSON (sorted keys, no whitespace variance,
no timestamps) and `hash` prints its SHA-256, so two lowerings are the same
schedule exactly when their hashes match.
"""
import argparse
import hashlib
import json
import os
import sys
import time
from collections import Counter

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

import decode_megakernel_02_gb300 as mk  # noqa: E402


def lower(workload, sms=152, chunks=0):
    """The IR of a synthetic workload's lowering on `sms` CTAs (plain Python data)."""
    w = synthetic.get_workload(workload)
    return mk.mk_build_ir(mk.make_desc(w), mk.make_config(sms=sms, attn_chunks=chunks), sms)


def canonical(ir):
    """The IR as canonical JSON text: the deterministic schedule artifact."""
    doc = {
        "n_sms": ir["n_sms"], "n_counters": ir["n_counters"], "n_buffers": ir["n_buffers"],
        "outputs": sorted(ir["outputs"]),
        "tagged": {str(c): b for c, b in sorted(ir.get("tagged", {}).items())},
        "tasks": [{"sm": t["sm"], "op": t.get("op", 0), "layer": t.get("layer", 0),
                   "waits": [list(x) for x in t["waits"]], "signal": t["signal"],
                   "acc": [list(a) for a in t["acc"]]} for t in ir["tasks"]],
        "queues": ir["queues"],
    }
    return json.dumps(doc, sort_keys=True, separators=(",", ":"))


def from_canonical(text):
    """Inverse of canonical(): an IR dict that mk_validate_ir accepts."""
    doc = json.loads(text)
    return {
        "n_sms": doc["n_sms"], "n_counters": doc["n_counters"], "n_buffers": doc["n_buffers"],
        "outputs": doc["outputs"], "tagged": {int(c): b for c, b in doc["tagged"].items()},
        "tasks": [{"sm": t["sm"], "op": t["op"], "layer": t["layer"],
                   "waits": [tuple(x) for x in t["waits"]], "signal": t["signal"],
                   "acc": [tuple(a) for a in t["acc"]]} for t in doc["tasks"]],
        "queues": doc["queues"],
    }


def digest(ir):
    return hashlib.sha256(canonical(ir).encode()).hexdigest()


def explain(ir):
    """A summary of the schedule: tasks per instruction and layer, queue
    lengths, counters (and which are carried by tagged values), accesses."""
    ops = Counter(mk.OPS.get(t["op"], str(t["op"])) for t in ir["tasks"])
    layers = {t["layer"] for t in ir["tasks"] if mk.OPS.get(t["op"]) == "qkv"}
    qlen = [len(q) for q in ir["queues"]]
    waits = sum(len(t["waits"]) for t in ir["tasks"])
    return {
        "tasks": len(ir["tasks"]),
        "tasks_per_op": dict(sorted(ops.items())),
        "decoder_layers": len(layers),
        "ctas": ir["n_sms"],
        "queue_length": {"min": min(qlen), "max": max(qlen), "mean": round(sum(qlen) / len(qlen), 2)},
        "counters": ir["n_counters"],
        "tagged_counters": len(ir.get("tagged", {})),
        "waits": waits,
        "accesses": sum(len(t["acc"]) for t in ir["tasks"]),
        "sha256": digest(ir),
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("command", choices=["explain", "validate", "dump", "hash"])
    ap.add_argument("--workload", default="llama-1b")
    ap.add_argument("--sms", type=int, default=152)
    ap.add_argument("--chunks", type=int, default=0, help="split-KV chunks per KV head (0: default rule)")
    ap.add_argument("--ir", help="read the IR from a file written by `dump` instead of lowering")
    ap.add_argument("--out", help="dump: output file (default: stdout)")
    args = ap.parse_args(argv)

    mk.load()
    if args.ir:
        with open(args.ir) as f:
            ir = from_canonical(f.read())
    else:
        ir = lower(args.workload, args.sms, args.chunks)
    if args.command == "explain":
        print(json.dumps(explain(ir), indent=1))
    elif args.command == "hash":
        print(digest(ir))
    elif args.command == "dump":
        text = canonical(ir)
        if args.out:
            with open(args.out, "w") as f:
                f.write(text)
        else:
            print(text)
    else:
        t0 = time.perf_counter()
        st, why = mk.mk_validate_ir(ir)
        print(json.dumps({"status": "ok" if st == mk.MK_OK else "rejected", "why": why,
                          "seconds": round(time.perf_counter() - t0, 3)}))
        return 0 if st == mk.MK_OK else 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
