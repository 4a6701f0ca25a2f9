"""Shared helpers of the GPU parity tests (comparison rules)."""
import numpy as np

LOGIT_ATOL = 1e-2   # teacher-forced logits, absolute
TIE_GAP = 1e-2      # greedy tokens must match where the oracle's top-1/top-2 gap exceeds this


def check_greedy_against_oracle(gen, z_oracle, where=""):
    """gen: GPU tokens; z_oracle[i]: oracle logits that predict gen[i] (teacher forced on gen).
    Where the oracle's top-1/top-2 gap exceeds TIE_GAP the tokens must be identical; elsewhere the
    GPU token must be within TIE_GAP of the oracle's maximum."""
    n_strict = 0
    for i, tok in enumerate(gen):
        z = z_oracle[i]
        top2 = np.partition(z, -2)[-2:]
        gap = float(top2[1] - top2[0])
        best = int(np.argmax(z))
        if gap > TIE_GAP:
            n_strict += 1
            assert int(tok) == best, f"{where} step {i}: gpu {int(tok)} oracle {best} (gap {gap:.4f})"
        else:
            assert float(z[int(tok)]) >= float(top2[1]) - TIE_GAP, f"{where} step {i}: near tie violated"
    return n_strict


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))
