"""Run a handful of launches of one solver kernel on a synthetic workload.

Meant for profilers (a few launches, bounded memory):
  python -m temporal_blocked_jacobi_gb300.profile_case --n 8192 --r 100 \
      --source gauss --strategy etb8 --launches 4 --residuals 1
Strategy tokens: sync | syncu (unfused right-hand side) | etbD | baD |
baDoO (overlap O) | any of them with @TXxTY. Prints the mean launch time
measured with CUDA events on the solver's stream.
"""
from __future__ import annotations

import argparse

from . import problem as P


def main(argv=None):
    import torch

    from . import jacobi

    ap = argparse.ArgumentParser()
    ap.add_argument("--n", type=int, default=8192)
    ap.add_argument("--r", type=float, default=100.0)
    ap.add_argument("--source", default="gauss")
    ap.add_argument("--strategy", default="sync")
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--residuals", type=int, default=1)
    a = ap.parse_args(argv)

    tok, tile = a.strategy, (0, 0)
    if "@" in tok:
        tok, t = tok.split("@")
        tile = tuple(int(v) for v in t.lower().split("x"))
    if tok == "sync":
        kw = dict(strategy="sync", depth=1)
    elif tok == "syncu":  # unfused right-hand side
        kw = dict(strategy="sync", depth=1, rhs="unfused")
    elif tok.startswith("etb"):
        kw = dict(strategy="etb", depth=int(tok[3:]))
    elif tok.startswith("ba") and "o" in tok:  # baDoO: overlap O both ways
        depth, ov = tok[2:].split("o")
        kw = dict(strategy="ba", depth=int(depth), overlap=(int(ov), int(ov)))
    elif tok.startswith("ba"):
        kw = dict(strategy="ba", depth=int(tok[2:]))
    else:
        raise SystemExit(f"unknown strategy {a.strategy}")

    n = a.n
    ld = P.padded_ld(n)
    u0 = torch.from_numpy(P.initial_field(n, ld)).cuda()
    g = torch.from_numpy(P.source_term(n, ld, a.source)).cuda()
    u, u_alt, b = jacobi.allocate(n, ld)
    u.copy_(u0)
    stream = torch.cuda.current_stream()
    with jacobi.Solver(u, u_alt, b, a.r, tile=tile, **kw) as s:
        s.rhs(g)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s.sweeps(a.launches)
        end.record(stream)
        for _ in range(a.residuals):
            s.residual()
        end.synchronize()
        ms = start.elapsed_time(end) / max(a.launches, 1)
    print(f"n={n} strategy={a.strategy} launches={a.launches} mean_launch_ms={ms:.4f}")


if __name__ == "__main__":
    main()
