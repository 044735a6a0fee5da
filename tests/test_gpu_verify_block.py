"""Parity of dspark_verify_block (block verification: the block value of
rejection_sample_method in brb-nv/TensorRT-LLM PR #21, "2. Golden sampling
semantics", Sun et al. 2024) with the CPU oracle.

The kernel computes the weight chain with the oracle's float32 operations,
but sums r_i = sum_x max(w_i p_i(x) - q_i(x), 0) in float32 where the oracle
sums in double.  So accepted_len must be identical except for requests where
some uniform lies within H_TOL of its threshold h_i.  The emitted token must
be identical wherever accepted_len is, except where the oracle's two best
Gumbel-max scores lie within TOKEN_TIE of each other."""
import numpy as np
import pytest
import torch

import ancestral_draft_sampling_gb300 as pkg
import oracle
from ancestral_draft_sampling_gb300 import workloads as wl
from tests.parity import TOKEN_TIE

pytestmark = pytest.mark.gpu

H_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _u64(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int64)).cuda()


def _gpu(v, fn=pkg.verify_block):
    acc, emit = fn(torch.from_numpy(v.q).cuda(), torch.from_numpy(v.p).cuda(),
                   torch.from_numpy(v.tokens).cuda(), _u64(v.seed),
                   _u64(v.offset))
    torch.cuda.synchronize()
    return acc.cpu().numpy(), emit.cpu().numpy()


def _check(v, acc, emit, skip=()):
    keep = np.array([b for b in range(v.B) if b not in set(skip)])
    ref = oracle.verify_block(v.q[keep], v.p[keep], v.tokens[keep],
                              v.seed[keep], v.offset[keep])
    near = (np.abs(ref.eta.astype(np.float64) - ref.h) <= H_TOL).any(axis=1)
    same = acc[keep] == ref.accepted_len
    assert (same | near).all(), (
        f"accepted_len differs away from a threshold: rows "
        f"{keep[~(same | near)][:5]}")
    ties = 0
    for i, b in enumerate(keep):
        if not same[i] or emit[b] == ref.emitted[i]:
            continue
        gap = float(ref.top2[i, 0] - ref.top2[i, 1])
        assert gap <= TOKEN_TIE, (
            f"request {b}: gpu {emit[b]} oracle {ref.emitted[i]}, gap {gap}")
        ties += 1
    return ref, ties, int((~same).sum())


@pytest.mark.parametrize("B,K,V", [
    (12, 5, 5001),     # one CTA per request, ragged vocabulary
    (40, 3, 4096),     # one CTA per request, float4 loads
    (12, 5, 40000),    # clusters of 8 CTAs
    (12, 4, 40003),    # clusters of 8, ragged slices and a ragged last block
    (1, 1, 9000),      # one draft: no sums
    (3, 64, 1024),     # the largest K
    (300, 2, 20000),   # more requests than the GPU has SMs
])
def test_verify_block_matches_oracle(B, K, V):
    v = wl.make_verify(B, K, V, seed=B * 1000 + K + V + 7)
    acc, emit = _gpu(v)
    ref, ties, flips = _check(v, acc, emit)
    assert ties <= 1 and flips <= 1
    assert ((acc >= 0) & (acc <= K)).all()


def test_verify_block_branch_cases():
    B, K, V = 16, 4, 40000
    v = wl.make_verify(B, K, V, seed=191)
    rng = np.random.default_rng(192)
    for b in range(B):
        if b in (0, 1):
            v.p[b, :K] = v.q[b]          # draft equal to target: all accepted
        if b == 2:
            v.p[b, 1:K] = 0.0            # zero targets after the first draft
        if b == 3:
            idx = rng.choice(V, size=200, replace=False)
            v.q[b, :, idx[:100]] = np.nan
            v.p[b, :, idx[100:]] = np.nan
        if b == 4:
            v.q[b, 0, v.tokens[b, 0]] = 0.0  # the draft had no draft mass
        if b == 5:
            v.p[b, K, :] = 0.0           # all-zero bonus row
            v.p[b, :K] = v.q[b]
    acc, emit = _gpu(v)
    ref, ties, flips = _check(v, acc, emit)
    assert ties == 0 and flips == 0
    assert acc[0] == K and acc[1] == K
    assert acc[5] == K and emit[5] == 0


def test_verify_block_invalid_draft_marks_only_that_request():
    v = wl.make_verify(6, 3, 9000, seed=15)
    v.tokens[1, 2] = 9000
    v.tokens[3, 0] = -7
    acc, emit = _gpu(v)
    assert acc[1] == -1 and emit[1] == -1
    assert acc[3] == -1 and emit[3] == -1
    _check(v, acc, emit, skip=(1, 3))


def test_verify_block_deterministic():
    v = wl.make_verify(24, 5, 30000, seed=27)
    a1 = _gpu(v)
    a2 = _gpu(v)
    np.testing.assert_array_equal(a1[0], a2[0])
    np.testing.assert_array_equal(a1[1], a2[1])


def test_verify_block_full_size_accepts_more_than_standard():
    # the verification that follows the B=88, K=7, V=200064 draft block
    v = wl.make_verify(88, 7, 200064, seed=1004, logit_std=4.0)
    acc, emit = _gpu(v)
    ref, ties, flips = _check(v, acc, emit)
    assert ties <= 1 and flips <= 1
    std, _ = _gpu(v, pkg.verify_standard)
    assert acc.mean() >= std.mean()
