"""Batch invariance of the core attention (report §3.3: the output of a given
token must not depend on the batch it is computed in).

With CSA_ATTEND_BATCH_INVARIANT a query's item list is cut into splits whose
number and boundaries depend only on its own item count, and the splits are
merged in a fixed order, so the same query must give bitwise the same output
and lse whether it is computed alone, with a few others, or in a batch of 32.
The outputs are also checked against the oracle."""
import numpy as np
import pytest
import torch

from long_context_sparse_21_b300 import abi, synth
from oracle import codecs, csa

from helpers import f64, max_abs_rel

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True, scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    abi.lib()


def _setup(seed, ctx, m, k):
    B = len(ctx)
    s = synth.Synth(seed, DEV)
    nk = max(c + 1 for c in ctx) // m
    ent = s.normal("entries", (B, nk, 576))
    pool = abi.make_pool(abi.FMT_KV_POOL_FP8, B, nk, 576, page_entries=256, device=DEV, shuffle_seed=seed)
    abi.csa_cache_write(ent, pool)
    ring = s.normal("ring", (B, 128, 576), dtype=torch.bfloat16)
    q = s.normal("q", (B, 64, 576), dtype=torch.bfloat16)
    pos = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    rows, cnts = [], []
    gen = np.random.Generator(np.random.Philox(synth._key(seed, "sel")))
    for t in ctx:
        nc = (t + 1) // m
        kk = min(k, nc)
        r = np.full(k, -1, np.int32)
        r[:kk] = np.sort(gen.choice(nc, size=kk, replace=False))
        rows.append(r)
        cnts.append(kk)
    idx = torch.tensor(np.array(rows), device=DEV)
    cnt = torch.tensor(cnts, dtype=torch.int32, device=DEV)
    return ent, pool, ring, q, pos, idx, cnt


CASES = {
    # CSA decode shape: 512 selected entries + 128 window rows = 20 tiles -> 4 splits
    "csa": dict(sparse=True, m=4, k=512, ctx=[8000 + 37 * b for b in range(32)]),
    # dense (HCA-style) over 1250-5000 entries: 44-161 tiles -> up to 8 splits, one cluster of 8
    "dense": dict(sparse=False, m=4, k=0, ctx=[5000 + 473 * b for b in range(32)]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_attend_bitwise_equal_across_batches(name):
    c = CASES[name]
    ctx, m, k, sparse = c["ctx"], c["m"], c["k"], c["sparse"]
    ent, pool, ring, q, pos, idx, cnt = _setup(51, ctx, m, max(k, 1))
    B = len(ctx)
    full = abi.AttendCall(sparse, q, pos, pool, 128, ring, 1 / 24, m, max(ctx), B, idx=idx, cnt=cnt,
                          batch_invariant=True)
    o_all, l_all = full()
    torch.cuda.synchronize()
    assert full.status() == abi.OK
    assert full.plan()[1] in (0, 1)  # split in a cluster (or not at all)
    o_all, l_all = o_all.clone(), l_all.clone()
    # the same queries alone (batch of one query), and in a batch of five in another order
    for rows in ([0], [7], [31], [3, 0, 31, 7, 12]):
        sel = torch.tensor(rows, dtype=torch.long, device=DEV)
        seq = sel.to(torch.int32)
        sub = abi.AttendCall(sparse, q[sel].contiguous(), pos[sel].contiguous(), pool, 128, ring, 1 / 24, m,
                             int(pos[sel].max()), B, idx=idx[sel].contiguous(), cnt=cnt[sel].contiguous(), seq=seq,
                             batch_invariant=True)
        o, l = sub()
        torch.cuda.synchronize()
        assert sub.status() == abi.OK
        for i, b in enumerate(rows):
            assert torch.equal(o[i], o_all[b]), (name, rows, b)
            assert torch.equal(l[i], l_all[b]), (name, rows, b)
    # and the batch's outputs are right
    entn = ent.cpu().numpy()
    ringn = f64(ring)
    for b in (0, 31):
        t = ctx[b]
        sel_rows = idx[b, : int(cnt[b])].cpu().numpy() if sparse else np.arange((t + 1) // m)
        X = codecs.kv_entry_decode(*codecs.kv_entry_encode(entn[b, sel_rows]))
        wp = csa.window_positions(t, 128)
        wo, wl = csa.attend_one(f64(q[b]), X, ringn[b, wp % 128], 1 / 24)
        assert max_abs_rel(f64(o_all[b]), wo) <= 2e-2
        assert np.allclose(f64(l_all[b]), wl, atol=2e-2)
