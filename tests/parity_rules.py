"""Comparison rules between the CUDA path and the oracle (test helpers only).

Tolerance (per row r, absolute plus relative to the row's largest logit):
    tol_r = 1e-3 * (1 + max_v |logit[r, v]|)
Rules:
  * given identical float32 logits: top-k ids and values bit-exact; draft ids
    exact wherever the oracle's walk margin exceeds a tight bound;
  * scores (unary and lattice): |gpu - oracle| <= tol_r;
  * fused LM-head path: candidate sets equal up to swaps of tokens whose oracle
    logits lie within tol_r of the oracle's k-th logit; draft ids compared along
    each sequence while its candidates match and every walk margin exceeds tol_r.
"""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def row_tol(ora_logits: np.ndarray) -> np.ndarray:
    return 1e-3 * (1.0 + np.abs(ora_logits).max(axis=1).astype(np.float64))


def check_sorted_lists(ids: np.ndarray, vals: np.ndarray) -> None:
    """Each row is sorted by (value desc, id asc) with distinct ids."""
    for r in range(ids.shape[0]):
        assert len(set(ids[r].tolist())) == ids.shape[1], f"row {r}: repeated candidate"
        for j in range(ids.shape[1] - 1):
            a, b = vals[r, j], vals[r, j + 1]
            assert a > b or (a == b and ids[r, j] < ids[r, j + 1]), f"row {r}: order broken at {j}"


def check_fused_candidates(gpu_ids, gpu_vals, ora_logits, ora_ids, ora_vals, tol):
    """Candidate sets match up to near-tie swaps; unary scores within tol. Returns the swap count."""
    R, k = gpu_ids.shape
    check_sorted_lists(gpu_ids, gpu_vals)
    swaps = 0
    for r in range(R):
        kth = float(ora_vals[r, k - 1])
        G, O = set(gpu_ids[r].tolist()), set(ora_ids[r].tolist())
        for g in G - O:
            assert ora_logits[r, g] >= kth - tol[r], f"row {r}: token {g} is not near the top-{k} boundary"
        for o in O - G:
            assert ora_logits[r, o] <= kth + tol[r], f"row {r}: dropped token {o} was clearly inside the top-{k}"
        swaps += len(G - O)
        err = np.abs(gpu_vals[r].astype(np.float64) - ora_logits[r, gpu_ids[r]].astype(np.float64))
        assert np.all(err <= tol[r]), f"row {r}: unary score error {err.max()} > {tol[r]}"
    return swaps


def compare_lattice_and_draft(gpu_lat, gpu_draft, ora, T, k, tol, margin_floor=None, stats=None):
    """Lattice scores where candidates agree; draft along each sequence while comparable.

    A step whose oracle walk margin is at or below the floor (a near tie that float32
    rounding may decide either way) is counted as low-margin: if both sides still chose the
    same candidate the sequence goes on (the next row reads the same predecessor row),
    otherwise the paths part there and the rest of the sequence is not comparable.
    Returns (compared_steps, low_margin_steps); `stats` (a dict) also receives
    'agreed_low', 'parted' and 'unreached' counts."""
    B = gpu_draft.shape[0]
    R = B * T
    gpu_ids = gpu_lat[:, :k].astype(np.int64)
    ora_ids = ora["topk_ids"].astype(np.int64)
    assert np.all(gpu_lat[:, :k] == np.floor(gpu_lat[:, :k])), "candidate ids are not exact floats"
    same = np.all(gpu_ids == ora_ids, axis=1)
    gs = gpu_lat[:, k:].reshape(R, k, k).astype(np.float64)
    os_ = ora["lattice"][:, k:].reshape(R, k, k).astype(np.float64)
    for r in range(R):
        t = r % T
        prev_same = True if t == 0 else same[r - 1]
        if same[r] and prev_same:
            err = np.abs(gs[r] - os_[r]).max()
            assert err <= tol[r], f"row {r}: lattice error {err} > {tol[r]}"
        if t == 0:
            assert np.all(gs[r] == gs[r][0:1]), f"row {r}: position-0 predecessor rows differ"
    compared, low, agreed_low, parted, unreached = 0, 0, 0, 0, 0
    floor = tol if margin_floor is None else margin_floor
    for b in range(B):
        for t in range(T):
            r = b * T + t
            if not same[r] or (t > 0 and not same[r - 1]):
                unreached += T - t
                break
            if ora["margins"][b, t] <= floor[r]:
                low += 1
                if gpu_draft[b, t] == ora["draft"][b, t]:
                    agreed_low += 1
                    continue
                parted += 1
                unreached += T - t - 1
                break
            assert gpu_draft[b, t] == ora["draft"][b, t], f"sequence {b} position {t}: draft differs"
            compared += 1
    if stats is not None:
        stats.update(compared=compared, low=low, agreed_low=agreed_low, parted=parted, unreached=unreached)
    return compared, low


# One line per full-size comparison, printed at the end of the pytest run (conftest).
REPORT = []


def report(line: str) -> None:
    REPORT.append(line)
