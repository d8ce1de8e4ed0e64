"""GPU-vs-oracle comparison rules.

 - candidate lists (top-128 ids in order): bit-exact;
 - greedy tokens, accept/reject decisions, num_kept and status words:
   bit-exact, except where the oracle reports the deciding floating-point
   comparison within a stated margin of its threshold ("ambiguous");
 - stochastic tokens: bit-exact wherever the two best perturbed scores differ
   by more than 1e-5 relative;
 - kept probabilities: within 1e-5 absolute.

Margins: top-p / min-p cut points and accept tests of truncated rows are
decided in fp64 on both sides (ambiguous below 1e-9); the accept test of an
untruncated row uses the full-vocabulary normaliser, which the kernels
accumulate in fp32 per tile (ambiguous below 1e-5 relative); Gumbel argmaxes
are decided in fp32 on both sides (ambiguous below 1e-5 relative, the
tolerance of the specification).
"""
from __future__ import annotations

import numpy as np

CUT_TOL = 1e-9
ACCEPT_TOL_TRUNC = 1e-9
ACCEPT_TOL_FULL = 1e-5
GUMBEL_TOL = 1e-5
PROB_TOL = 1e-5

GREEDY = 1
TOPK, TOPP, MINP, BOUNDED_P = 16, 32, 64, 128


def _trunc(rows, r):
    f = int(rows["flags"][r])
    if f & GREEDY:
        return False
    return bool(((f & TOPK) and rows["top_k"][r] > 0) or ((f & TOPP) and rows["top_p"][r] < 1)
                or ((f & MINP) and rows["min_p"][r] > 0) or (f & BOUNDED_P))


class Report:
    def __init__(self):
        self.checked = 0
        self.ambiguous = 0
        self.errors = []

    def fail(self, msg):
        if len(self.errors) < 20:
            self.errors.append(msg)

    def ok(self):
        return not self.errors

    def __repr__(self):
        return f"Report(checked={self.checked}, ambiguous={self.ambiguous}, errors={self.errors[:8]})"


def compare_candidates(rep: Report, gpu: dict, ora: dict, positions):
    for p in positions:
        a, b = gpu["cand_ids"][p], ora["cand_ids"][p]
        if not np.array_equal(a, b):
            k = int(np.argmax(a != b))
            rep.fail(f"pos {p}: cand_ids differ at {k}: gpu {a[k]} oracle {b[k]}")
            continue
        na, nb = int(gpu["num_kept"][p]), int(ora["num_kept"][p])
        if na != nb:
            if min(ora["margin_topp"][p], ora["margin_minp"][p]) < CUT_TOL:
                rep.ambiguous += 1
                continue
            rep.fail(f"pos {p}: num_kept gpu {na} oracle {nb} (margins {ora['margin_topp'][p]:.3g}, "
                     f"{ora['margin_minp'][p]:.3g})")
            continue
        d = np.max(np.abs(gpu["cand_probs"][p] - ora["cand_probs"][p]))
        if d > PROB_TOL:
            rep.fail(f"pos {p}: cand_probs differ by {d:.3g}")
        rep.checked += 1


def compare_sample(w, gpu: dict, ora: dict, rows=None) -> Report:
    rep = Report()
    rows = range(w.B) if rows is None else rows
    compare_candidates(rep, gpu, ora, rows)
    for r in rows:
        tg, to = int(gpu["tokens"][r]), int(ora["tokens"][r])
        sg, so = int(gpu["row_status"][r]), int(ora["row_status"][r])
        if sg != so:
            rep.fail(f"row {r}: status gpu {sg:#x} oracle {so:#x}")
        if tg != to:
            amb = ora["margin_gumbel"][r] < GUMBEL_TOL or min(ora["margin_topp"][r], ora["margin_minp"][r]) < CUT_TOL
            if amb:
                rep.ambiguous += 1
            else:
                rep.fail(f"row {r}: token gpu {tg} oracle {to} (gumbel margin {ora['margin_gumbel'][r]:.3g})")
        rep.checked += 1
    return rep


def compare_verify(w, gpu: dict, ora: dict, rows=None) -> Report:
    rep = Report()
    rows = range(w.B) if rows is None else rows
    offs = w.position_offsets()
    gam = w.gammas()
    positions = [p for r in rows for p in range(int(offs[r]), int(offs[r]) + int(gam[r]) + 1)]
    compare_candidates(rep, gpu, ora, positions)
    for r in rows:
        na, nb = int(gpu["num_accepted"][r]), int(ora["num_accepted"][r])
        ta, tb = gpu["tokens"][r], ora["tokens"][r]
        sg, so = int(gpu["row_status"][r]), int(ora["row_status"][r])
        if na == nb and np.array_equal(ta, tb) and sg == so:
            rep.checked += 1
            continue
        # the walks first differ at min(na, nb)
        j = min(na, nb)
        p = int(offs[r]) + j
        acc_tol = ACCEPT_TOL_TRUNC if _trunc(w.rows, r) else ACCEPT_TOL_FULL
        amb = (ora["margin_accept"][p] < acc_tol or ora["margin_resid"][p] < GUMBEL_TOL
               or ora["margin_gumbel"][p] < GUMBEL_TOL
               or min(ora["margin_topp"][p], ora["margin_minp"][p]) < CUT_TOL)
        if amb:
            rep.ambiguous += 1
        else:
            rep.fail(f"row {r}: gpu acc {na} tok {ta.tolist()} st {sg:#x} | oracle acc {nb} tok {tb.tolist()} "
                     f"st {so:#x} (pos {p}: acc margin {ora['margin_accept'][p]:.3g}, resid "
                     f"{ora['margin_resid'][p]:.3g}, gumbel {ora['margin_gumbel'][p]:.3g})")
        rep.checked += 1
    return rep
