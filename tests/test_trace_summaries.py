"""The summaries the profiling hook's stamps are reduced to
(attention_forward_online_gb300/run_workload.py: print_step_trace,
print_cta_times), checked on synthetic stamps whose phase lengths are known:
the per-step and per-CTA tables of the forward profiles come from these two
functions."""
import numpy as np

from attention_forward_online_gb300.run_workload import print_cta_times, print_step_trace


def synthetic_steps(n=20, step=3000):
    tr = np.zeros((8, 7, 128, 4), dtype=np.int64)
    for j in range(n):
        t = 10_000 + step * j
        tr[0, 0, j] = [t, t + 50, t + 450, t + 1350]                 # S seen, loaded, alpha, P
        tr[0, 3, j] = [t + 1350, t + 1440, t + 1250, t + 1260]       # P published, per warp
        tr[0, 5, j] = [t + 500, t + 900, t + 950, j % 2]             # correction of tile 0
        tr[0, 2, j, 0] = t - 100                                     # MMA iteration start
    for j in range(1, n):
        t_prev = 10_000 + step * (j - 1)
        tr[0, 2, j, 1] = t_prev + 1440 + 80                          # MMA sees P of step j - 1
    return tr


def test_step_summary_recovers_the_phases(capsys):
    # steps 2 .. n-2 are summarised: 17 of 20, 8 of them with the rescale flag
    print_step_trace(synthetic_steps())
    out = capsys.readouterr().out
    assert ("CTA 0: 20 steps; cycles per K/V step 3000; softmax of tile 0: S load 50, "
            "row max + alpha 400, P 900 (busy 1350); P published -> next S seen (PV + S) 1650; "
            "MMA issuer iteration 3000") in out
    assert ("softmax warps publish P at +90 / -100 / -90 cycles from its first warp; "
            "correction arrives -490 from the last of them and rescaled O in 47 % of steps; "
            "last arrival -> MMA warp sees P 80") in out
    # CTAs without enough steps are skipped
    assert "CTA 1" not in out


def test_cta_summary_recovers_the_phases(capsys):
    ct = np.zeros((4096, 6), dtype=np.int64)
    #            start  setup  first S  epilogue  end    SM
    ct[0] = [0, 500, 2000, 9000, 10_000, 0]
    ct[1] = [0, 500, 2000, 9000, 10_000, 1]
    ct[2] = [11_000, 11_500, 13_000, 20_000, 21_000, 0]
    ct[3] = [12_000, 12_500, 14_000, 21_000, 22_000, 1]
    print_cta_times(ct, 4)
    out = capsys.readouterr().out
    assert ("CTAs 4 on 2 SMs over 22.0 us; per CTA (median, us): setup 0.50, to the first S 1.50, "
            "K/V loop 7.00, epilogue 1.00; gap between CTAs on an SM 1.50; SMs busy 0.909") in out
