"""Probability mass outside the top-128 candidates on the standard
workloads, from the oracle: per target position, 1 minus the full-vocabulary
softmax mass of its 128 candidates, at the row's temperature after the
logits processors (greedy rows at T = 1).  This is the synthetic stand-in
for the SonicSampler pages' claim (section 1) that the top 128 hold nearly
all of the relevant mass.

    python -m tests.mass_report
"""
import numpy as np

from oracle import oracle
from spec_verification_gb300 import workloads as W


def mass_outside(w) -> np.ndarray:
    out = oracle.verify(w) if w.is_verify else oracle.sample(w)
    return np.asarray(out["mass_outside"], np.float64)


def summary(m: np.ndarray) -> str:
    return (f"{m.size} positions: min {m.min():.3g}, median {np.median(m):.3g}, "
            f"max {m.max():.3g}")


if __name__ == "__main__":
    for name, make in [("c1", W.config1), ("c2", W.config2), ("c3", W.config3), ("c4", W.config4),
                       ("c5", W.config5)]:
        w = make()
        m = mass_outside(w)
        print(f"{name}: {summary(m)}")
        if name == "c3":
            half = w.B // 2
            print(f"  c3 Zipf-boosted rows: {summary(m[:half])}")
            print(f"  c3 near-flat rows:    {summary(m[half:])}")
