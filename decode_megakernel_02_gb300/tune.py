"""Grid search over the schedule knobs.

AutoMegaKernel explainer, "Methodology" (Layer 2 scheduler, autoresearch
loop): change the ScheduleConfig, validate it, check the result, time it, and
keep the fastest.  This is the deterministic core of that loop, with no agent:

1. Every grid point goes through the static validator (`mk_validate_schedule`).
   A rejected schedule is recorded with its reason and never launched.
2. Each accepted point decodes the same teacher-forced token stream. Its logits
   must match the reference: max|dlogit| <= 1e-2 * max|logit| per step, with
   the same argmax on >= 99% of the steps.  The reference is a file of
   teacher-forced logits given with --reference (float32 [forced, vocab], the
   logits of the last prompt token and of forced tokens 1.. of the stream
   `forced_stream` builds; the parity tests write it from the CPU oracle), or,
   without one, the default configuration's own logits.
3. The points that pass are timed with CUDA events over full decode launches.
   The result is printed as JSON, fastest first.

    python -m decode_megakernel_02_gb300.tune --workload llama-1b --chunks 2,3,4,6,8 --sms 0,144
"""
import itertools
import argparse
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

import decode_megakernel_02_gb300 as mk  # noqa: E402

TOL = 1e-2


def agrees(lg, ref, tol=TOL):
    """Per-step max|dlogit| <= tol * max|ref| and >= 99% argmax agreement."""
    if lg.shape != ref.shape or not np.all(np.isfinite(lg)):
        return False
    for s in range(ref.shape[0]):
        if np.abs(lg[s] - ref[s]).max() > tol * np.abs(ref[s]).max():
            return False
    return float(np.mean(lg.argmax(axis=1) == ref.argmax(axis=1))) >= 0.99


def run_point(desc, blob, cfg, prompt, forced, n_time, reps):
    """Teacher-forced logits and the mean launch time of an n_time-token decode."""
    import torch
    dec = mk.Decoder(desc, blob, cfg)
    try:
        dec.prefill(prompt)
        lg, _ = dec.teacher_forced(forced)
        ids = torch.empty(n_time, dtype=torch.int32, device="cuda")
        pos0, tok = len(prompt) - 1, int(prompt[-1])
        times = []
        for r in range(reps + 2):
            dec.set_state(pos0, tok)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(dec.stream)
            dec.decode_async(n_time, out_ids=ids)
            b.record(dec.stream)
            dec.finish()
            if r >= 2:
                times.append(a.elapsed_time(b))
        return lg, float(np.mean(times)), dec.launch_info()
    finally:
        dec.close()


def forced_stream(w, n):
    """Teacher-forced inputs: the last prompt token, then n - 1 seeded random tokens."""
    prompt = synthetic.generate_prompt(w)
    return prompt, np.concatenate([prompt[-1:], synthetic.gen.random_tokens(w, n - 1, 7)]).astype(np.int32)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama-1b")
    ap.add_argument("--chunks", default="0,2,3,4,6,8", help="split-KV chunks per KV head (0: default rule)")
    ap.add_argument("--sms", default="0", help="CTAs (0: every SM)")
    ap.add_argument("--forced", type=int, default=8, help="teacher-forced steps of the agreement check")
    ap.add_argument("--tokens", type=int, default=0, help="tokens per timed launch (default: the workload's)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--token-select", default="0", help="0 / 1: schedules with the token-select task")
    ap.add_argument("--reference", default=None, help=".npy teacher-forced reference logits [forced, vocab]")
    args = ap.parse_args(argv)

    from decode_megakernel_02_gb300 import build
    build.build()
    w = synthetic.get_workload(args.workload)
    weights = synthetic.generate_weights(w)
    desc = mk.make_desc(w)
    blob = mk.pack_model(desc, weights)
    del weights
    prompt, forced = forced_stream(w, args.forced)
    n_time = args.tokens or w.decode_steps

    if args.reference:
        ref, ref_kind = np.load(args.reference), "reference file"
        if ref.shape != (args.forced, w.vocab):
            raise SystemExit(f"--reference holds {ref.shape}, expected {(args.forced, w.vocab)}")
    else:
        ref, ref_kind = run_point(desc, blob, mk.make_config(), prompt, forced, 1, 1)[0], "default configuration"
    ints = (lambda v: [int(x) for x in v.split(",")])
    rows = []
    for sms, ch, ts in itertools.product(ints(args.sms), ints(args.chunks), ints(args.token_select)):
        cfg = mk.make_config(sms=sms, attn_chunks=ch, token_select=ts)
        point = {"sms": sms, "attn_chunks": ch, "token_select": ts}
        st, why = mk.mk_validate_schedule(desc, cfg, sms or 152)
        if st != mk.MK_OK:
            rows.append(dict(point, status="rejected by the validator", why=why))
            continue
        try:
            lg, ms, info = run_point(desc, blob, cfg, prompt, forced, n_time, args.reps)
        except mk.MKError as e:
            rows.append(dict(point, status="error", why=str(e)))
            continue
        if not agrees(lg, ref):
            rows.append(dict(point, status=f"rejected: logits differ from the {ref_kind}"))
            continue
        rows.append(dict(point, status="ok", tokens_per_s=n_time / (ms / 1000.0), ms_per_launch=ms,
                         ctas=info["ctas"], n_tasks=info["n_tasks"]))
    rows.sort(key=lambda r: -r.get("tokens_per_s", 0.0))
    print(json.dumps({"workload": w.name, "tokens_per_launch": n_time, "agreement_reference": ref_kind,
                      "points": rows}, indent=1))


if __name__ == "__main__":
    main()
