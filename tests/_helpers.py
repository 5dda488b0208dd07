"""Shared helpers for the oracle's statistical pins (CPU only)."""
import numpy as np


def logits_from_probs(p):
    """float32 logits whose softmax is p (zero probability -> -inf)."""
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p).astype(np.float32)


def sample_rows(rng, probs):
    """One categorical draw per row of probs [..., V] (numpy RNG, independent of Philox)."""
    probs = np.asarray(probs, dtype=np.float64)
    flat = probs.reshape(-1, probs.shape[-1])
    cdf = np.cumsum(flat, axis=1)
    cdf /= cdf[:, -1:]
    u = rng.random(flat.shape[0])
    idx = (u[:, None] > cdf).sum(axis=1)
    return np.minimum(idx, flat.shape[1] - 1).reshape(probs.shape[:-1]).astype(np.int32)


def chisq_pvalue(observed, expected_probs, min_expected=5.0):
    """Pearson chi-square p-value, pooling cells with small expectation."""
    from scipy import stats
    observed = np.asarray(observed, dtype=np.float64)
    n = observed.sum()
    exp = np.asarray(expected_probs, dtype=np.float64) * n
    big = exp >= min_expected
    obs_c = list(observed[big])
    exp_c = list(exp[big])
    if (~big).any():
        obs_c.append(observed[~big].sum())
        exp_c.append(exp[~big].sum())
    obs_c, exp_c = np.array(obs_c), np.array(exp_c)
    keep = exp_c > 0
    return stats.chisquare(obs_c[keep], exp_c[keep] * obs_c[keep].sum() / exp_c[keep].sum()).pvalue
