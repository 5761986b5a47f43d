"""Run libosattn on one workload a fixed number of times (for profilers).

    python -m attention_forward_online_gb300.run_workload --workload NAME
        [--launches N] [--heads H] [--step-trace]

Inputs are the seeded synthetic tensors of the named workload, resident on
cuda:0 before the first launch; --heads keeps only the first H heads (a
smaller case of the same kernel for detailed Nsight Compute captures).  A
backward workload runs the forward pass once, untimed, and then times the
backward call (its three kernels).  A row-softmax workload runs
osattn_softmax_rows (--heads then keeps that many thousand rows).  Prints
the median launch time from CUDA events on the launching stream.

--step-trace builds and loads the profiling library (the forward kernel's
per-step SM clock stamps compiled in, libosattn_trace.so) and prints, for
the first CTAs of the last launch, the steady-state cycles per K/V step and
how each role spends them.
"""
import argparse
import dataclasses
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    from attention_forward_online_gb300 import osattn
    from attention_forward_online_gb300.inputs import (BWD_WORKLOADS, ROW_WORKLOADS,
                                                       SPLITKV_WORKLOADS, WORKLOADS,
                                                       make_grad_out, make_inputs, make_rows)

    allw = dict(WORKLOADS, **SPLITKV_WORKLOADS, **BWD_WORKLOADS, **ROW_WORKLOADS)
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", required=True, choices=sorted(allw))
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--heads", type=int, default=0)
    ap.add_argument("--step-trace", action="store_true",
                    help="profile the forward kernel's K/V steps (profiling build)")
    ap.add_argument("--splits", type=int, default=-1,
                    help="key ranges for the split-KV entry point (0: unsplit; default: the workload's)")
    args = ap.parse_args(argv)
    if args.step_trace:
        from attention_forward_online_gb300 import _build

        osattn.LIB_PATH = _build.build(step_trace=True)
    w = allw[args.workload]
    if args.workload in ROW_WORKLOADS:
        return run_rows(w, args)
    if args.splits >= 0:
        w = dataclasses.replace(w, splits=args.splits)
    if args.heads:
        w = dataclasses.replace(w, H=min(args.heads, w.H))
    q, k, v, kl = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    kld = None if kl is None else kl.to(dev)
    O = torch.empty_like(qd)
    L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream(device=dev)
    ws = None
    if w.splits:
        ws = torch.empty(osattn.splitkv_workspace_bytes(w.B, w.H, w.Nq, w.d, w.splits),
                         dtype=torch.uint8, device=dev)
    if w.bwd:
        dod = make_grad_out(w).to(dev)
        osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal, key_len=kld, out=O, lse=L, stream=s)
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        ws = torch.empty(osattn.bwd_workspace_bytes(w.B, w.H, w.Nq), dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.launches)]
    flops = w.bwd_flops if w.bwd else w.flops
    with torch.cuda.stream(s):
        for i in range(args.launches):
            ev[2 * i].record(s)
            if w.bwd:
                osattn.bwd(qd, kd, vd, O, L, dod, scale=w.scale, causal=w.causal, key_len=kld,
                           dq=dq, dk=dk, dv=dv, workspace=ws, stream=s)
            elif w.splits:
                osattn.fwd_splitkv(qd, kd, vd, w.splits, scale=w.scale, causal=w.causal,
                                   key_len=kld, out=O, lse=L, workspace=ws, stream=s)
            else:
                osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal, key_len=kld, out=O,
                           lse=L, stream=s)
            ev[2 * i + 1].record(s)
    s.synchronize()
    st = osattn.get_device_status(s)
    if st != osattn.OK:
        print("device status:", osattn.status_string(st))
        return 1
    ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.launches)]
    med = sorted(ms[1:] if len(ms) > 1 else ms)[len(ms[1:] if len(ms) > 1 else ms) // 2]
    print(f"{w.name} H={w.H} splits={w.splits}: launches {args.launches}, median {med:.4f} ms = "
          f"{flops / (med * 1e-3) / 1e12:.1f} TFLOPS (first launch excluded); "
          f"ms {['%.4f' % m for m in ms]}")
    if args.step_trace:
        steps, ctas = osattn.step_trace()
        print_step_trace(steps)
        print_cta_times(ctas, grid_ctas(w))
    return 0


def print_step_trace(tr):
    """Steady-state summary of the forward kernel's per-step clock stamps
    (tr [cta, role, step, stamp], see osattn_step_trace_read): the steps
    after the first two and before the last of each traced CTA."""
    import numpy as np

    for cta in range(tr.shape[0]):
        sm0, sm1, mma = tr[cta, 0], tr[cta, 1], tr[cta, 2]
        n = int((sm0[:, 3] > 0).sum())
        if n < 6:
            continue
        js = np.arange(2, n - 1)
        step = np.diff(sm0[js, 0]).mean()
        ld = (sm0[js, 1] - sm0[js, 0]).mean()
        mx = (sm0[js, 2] - sm0[js, 1]).mean()
        pp = (sm0[js, 3] - sm0[js, 2]).mean()
        # from P published (step j) to S of step j+1 seen: the tile's MMAs
        mma_lat = (sm0[js[:-1] + 1, 0] - sm0[js[:-1], 3]).mean()
        mma_iter = np.diff(mma[js, 0]).mean()
        print(f"CTA {cta}: {n} steps; cycles per K/V step {step:.0f}; softmax of tile 0: "
              f"S load {ld:.0f}, row max + alpha {mx:.0f}, P {pp:.0f} "
              f"(busy {ld + mx + pp:.0f}); P published -> next S seen (PV + S) {mma_lat:.0f}; "
              f"MMA issuer iteration {mma_iter:.0f}")
        # P of tile 0 complete (last of the four softmax warps and the
        # correction warp) -> seen by the MMA warp; warp spread of P
        warps = tr[cta, 3][js]                       # [step, warp]
        corr = tr[cta, 5][js]                        # alpha seen, rescaled, arrived, flag
        last = np.maximum(warps.max(1), corr[:, 2])
        seen = mma[js + 1, 1] - last
        rel = (warps - warps[:, :1]).mean(0)
        print(f"       tile 0: softmax warps publish P at {rel[1]:+.0f} / {rel[2]:+.0f} / "
              f"{rel[3]:+.0f} cycles from its first warp; correction arrives "
              f"{(corr[:, 2] - warps.max(1)).mean():+.0f} from the last of them and rescaled O "
              f"in {100 * corr[:, 3].mean():.0f} % of steps; last arrival -> MMA warp sees P "
              f"{seen.mean():.0f}")


def grid_ctas(w):
    """CTAs of one bf16/fp16 forward launch: 256 query rows each (times the
    key ranges with split-KV)."""
    return w.B * w.H * ((w.Nq + 255) // 256) * max(1, getattr(w, "splits", 0) or 1)


def print_cta_times(ct, n):
    """Where each CTA's time goes (the profiling build's per-CTA global-timer
    stamps: start, setup done, first S seen, epilogue start, end, SM), over
    the first min(n, 4096) CTAs of the last launch, and how busy the SMs were
    between the first start and the last end."""
    import numpy as np

    ct = ct[:min(n, ct.shape[0])].astype(np.float64)
    ok = ct[:, 4] > 0
    ct = ct[ok]
    if len(ct) == 0:
        return
    start, setup, s0, epi, end, sm = (ct[:, i] for i in range(6))
    t0, t1 = start.min(), end.max()
    busy = sum((end[sm == s] - start[sm == s]).sum() for s in np.unique(sm))
    gaps = []
    for s in np.unique(sm):
        o = np.argsort(start[sm == s])
        st, en = start[sm == s][o], end[sm == s][o]
        gaps += list(st[1:] - en[:-1])
    med = lambda x: float(np.median(x)) / 1e3
    print(f"CTAs {len(ct)} on {len(np.unique(sm))} SMs over {(t1 - t0) / 1e3:.1f} us; per CTA "
          f"(median, us): setup {med(setup - start):.2f}, to the first S {med(s0 - setup):.2f}, "
          f"K/V loop {med(epi - s0):.2f}, epilogue {med(end - epi):.2f}; gap between CTAs on an "
          f"SM {med(gaps) if gaps else 0.0:.2f}; SMs busy {busy / (len(np.unique(sm)) * (t1 - t0)):.3f}")


def run_rows(w, args):
    import dataclasses

    import torch

    from attention_forward_online_gb300 import osattn
    from attention_forward_online_gb300.inputs import make_rows

    if args.heads:
        w = dataclasses.replace(w, rows=min(w.rows, 1000 * args.heads))
    xd = make_rows(w).to("cuda:0")
    yd = torch.empty_like(xd)
    ld = torch.empty(w.rows, dtype=torch.float32, device=xd.device)
    s = torch.cuda.Stream(device=xd.device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.launches)]
    with torch.cuda.stream(s):
        for i in range(args.launches):
            ev[2 * i].record(s)
            osattn.softmax_rows(xd, out=yd, lse=ld, stream=s)
            ev[2 * i + 1].record(s)
    s.synchronize()
    ms = sorted(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(1, args.launches))
    med = ms[len(ms) // 2] if ms else 0.0
    print(f"{w.name} rows={w.rows}: launches {args.launches}, median {med:.4f} ms = "
          f"{w.bytes_moved / (med * 1e-3) / 1e9:.0f} GB/s (first launch excluded)")
    return 0


if __name__ == "__main__":
    sys.exit(main())
