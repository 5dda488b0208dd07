"""Parity rules between the CUDA path and the oracle (shared by the GPU tests).

Rules (the verify step's stated tolerances):
  * greedy outputs are compared bit for bit;
  * sampled tokens and counts are compared bit for bit, except at a near-tie of
    the decision where the two first differ: an acceptance test with
    |u - p/q| < 1e-6, or a Gumbel-max draw whose top-2 keys (log w + g) are
    within 1e-6, both measured on the oracle's double-precision values;
    near-ties are counted and must stay under 1e-4 of all decisions;
  * p(x), q(x) and alpha agree within 1e-5 relative;
  * flags agree exactly;
  * with a nucleus (top-p) cut, a batch row whose oracle-reported nucleus gap is
    below 2e-6 counts as a near-tie where the outputs differ.
The opt-in inverse-transform sampler's tests pass their own draw window.
"""
import numpy as np

NEAR_TIE = 1e-6
NEAR_TIE_RATE = 1e-4
REL_TOL = 1e-5
# a nucleus (top-p) cut whose top_p lies this close to a cumulative probability
# at the cut may differ by that boundary group (fixed-point sums of fp32 exp2
# terms on the GPU, double on the oracle)
NEAR_NUCLEUS = 2e-6


def compare_sampling(gpu: dict, orc: dict, gamma: int, rows=None, check_pq=True,
                     near_draw=NEAR_TIE):
    """Returns (bad_rows, near_ties, decisions).  gpu: dict of numpy arrays.
    Decisions count every acceptance test taken and every draw."""
    B = orc["counts"].shape[0]
    rows = range(B) if rows is None else rows
    bad, near, decisions = [], 0, 0
    nuc = orc.get("nucleus_gap")
    for b in rows:
        no = int(orc["counts"][b])
        decisions += min(no + 1, gamma) + 1
        same = (int(gpu["counts"][b]) == no and
                np.array_equal(gpu["tokens"][b], orc["tokens"][b]))
        if (orc["flags"][b] & 2):  # non-finite rows: outputs unspecified, flags only
            same = True
        near_cut = nuc is not None and bool(nuc[b] < NEAR_NUCLEUS)
        if not same:
            ng = int(gpu["counts"][b])
            if not 0 <= ng <= gamma:
                is_near = False  # an out-of-range count is never a tie
            elif near_cut:
                is_near = True
            elif ng != no:
                j = min(ng, no)
                margin = abs(orc["u"][b, j] - orc["ratio"][b, j])
                is_near = bool(margin < NEAR_TIE)
            else:
                is_near = bool(orc["gap"][b] < near_draw)
            if is_near:
                near += 1
            else:
                bad.append(b)
        if int(gpu["flags"][b]) != int(orc["flags"][b]):
            bad.append(b)
        if check_pq and not (orc["flags"][b] & 2):
            for key in ("p", "q"):
                ref = orc[key][b]
                got = gpu[key][b].astype(np.float64)
                tol = REL_TOL * np.abs(ref) + 1e-37
                if not np.all(np.abs(got - ref) <= tol):
                    bad.append(b)
    return sorted(set(bad)), near, decisions


def describe(gpu, orc, b):
    return (f"row {b}: gpu tokens={gpu['tokens'][b].tolist()} n={gpu['counts'][b]} "
            f"flags={gpu['flags'][b]} | oracle tokens={orc['tokens'][b].tolist()} "
            f"n={orc['counts'][b]} flags={orc['flags'][b]} gap={orc['gap'][b]:.3e} "
            f"u={orc['u'][b].tolist()} ratio={orc['ratio'][b].tolist()} "
            f"p={orc['p'][b].tolist()} gpu_p={gpu['p'][b].tolist()}")


# (what, decisions, rows differing at a near-tie, near-ties in the oracle's own round)
RECORD = []


def record(what: str, decisions: int, near_differing: int, near_oracle: int):
    """Keep a config's counts for the end-of-session summary (tests/conftest.py)."""
    RECORD.append((what, int(decisions), int(near_differing), int(near_oracle)))


def to_np(d: dict) -> dict:
    return {k: (v.cpu().numpy() if hasattr(v, "cpu") else v) for k, v in d.items()}


def near_ties(orc: dict, gamma: int, rows=None) -> int:
    """Decisions of the oracle's own round that fall inside the near-tie rule
    (whether or not the GPU differs there)."""
    B = orc["counts"].shape[0]
    rows = range(B) if rows is None else rows
    n = 0
    for b in rows:
        k = int(orc["counts"][b])
        tested = min(k + 1, gamma)
        n += int(np.sum(np.abs(orc["u"][b, :tested] - orc["ratio"][b, :tested]) < NEAR_TIE))
        n += int(orc["gap"][b] < NEAR_TIE)
    return n


def assert_parity(gpu, orc, gamma, rows=None, check_pq=True, what="", near_draw=NEAR_TIE):
    bad, near, dec = compare_sampling(gpu, orc, gamma, rows, check_pq, near_draw)
    msg = "\n".join(describe(gpu, orc, b) for b in bad[:5])
    assert not bad, f"{what}: {len(bad)} rows differ beyond the near-tie rule\n{msg}"
    assert near <= NEAR_TIE_RATE * dec, f"{what}: {near} near-ties in {dec} decisions"
    return near, dec
