"""CPU checks of the test helpers that judge a kernel's selection: the
validity test against brute force over every (kept, dropped) pair, and the
score error bound against BF16 rounding done by torch."""
import numpy as np
import torch

from oracle import csa

from helpers import score_error_bound, selection_valid


def _brute(sel, cnt, scores, k, err):
    n = len(scores)
    if cnt != min(k, n):
        return False
    kept = set(int(x) for x in sel[:cnt])
    if len(kept) != cnt or any(x < 0 or x >= n for x in kept) or list(sel[:cnt]) != sorted(kept):
        return False
    if any(x != -1 for x in sel[cnt:]):
        return False
    e = np.broadcast_to(err, (n,))
    return all(scores[a] + e[a] >= scores[b] - e[b] for a in kept for b in range(n) if b not in kept)


def test_selection_valid_agrees_with_brute_force():
    rng = np.random.default_rng(5)
    for trial in range(400):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, 12))
        scores = np.round(rng.standard_normal(n) * 4) / 4
        err = rng.random(n) * 0.3 if trial % 2 else 0.1
        kk = min(k, n)
        sel = np.full(k, -1)
        if trial % 3 == 0:  # the exact top-k
            idx, c = csa.topk(scores, n, k)
            sel = idx
        else:  # a random subset, often invalid
            sel[:kk] = np.sort(rng.choice(n, kk, replace=False))
        ok, _ = selection_valid(sel, kk, scores, k, err)
        assert ok == _brute(sel, kk, scores, k, err), trial


def test_score_error_bound_covers_bf16_rounding():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((64, 128))
    w = rng.random(64)
    keys = rng.standard_normal((2000, 128))
    s = csa.index_scores(q, w, keys)
    s32 = torch.from_numpy(s.astype(np.float32))
    sb = s32.to(torch.bfloat16).float().numpy().astype(np.float64)
    e = score_error_bound(q, w, keys, bf16_scores=True)
    assert np.all(np.abs(sb - s) <= e)
    # and the bound is not vacuous: within a factor of a few of the worst rounding
    assert np.max(e / np.maximum(np.abs(s), 1e-30)) < 2.0 ** -6
