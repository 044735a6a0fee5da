"""Parity of dspark_verify_standard (the standard rule of brb-nv/TensorRT-LLM
PR #21, "2. Golden sampling semantics") with the CPU oracle.

accepted_len must be identical (the acceptance test is one float32 product
and compare on the same inputs on both sides).  The emitted token must be
identical except where the oracle's two best Gumbel-max scores lie within
TOKEN_TIE of each other.  Inputs come from the seeded generator, edited per
case to reach each branch of the rule: rejection with a residual draw, the
bonus draw after K acceptances, an all-zero residual (draw from p), an
all-zero drawing row, NaN and infinite probabilities, weights large enough
to leave the range of the kernel's candidate test, and invalid drafts."""
import numpy as np
import pytest
import torch

import ancestral_draft_sampling_gb300 as pkg
import oracle
from ancestral_draft_sampling_gb300 import workloads as wl
from tests.parity import TOKEN_TIE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _u64(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int64)).cuda()


def _gpu_verify(v):
    acc, emit = pkg.verify_standard(
        torch.from_numpy(v.q).cuda(), torch.from_numpy(v.p).cuda(),
        torch.from_numpy(v.tokens).cuda(), _u64(v.seed), _u64(v.offset))
    torch.cuda.synchronize()
    return acc.cpu().numpy(), emit.cpu().numpy()


def _check(v, acc, emit, skip=()):
    keep = np.array([b for b in range(v.B) if b not in set(skip)])
    ref = oracle.verify_standard(v.q[keep], v.p[keep], v.tokens[keep],
                                 v.seed[keep], v.offset[keep])
    np.testing.assert_array_equal(acc[keep], ref.accepted_len)
    ties = 0
    for i, b in enumerate(keep):
        if emit[b] != ref.emitted[i]:
            gap = float(ref.top2[i, 0] - ref.top2[i, 1])
            assert gap <= TOKEN_TIE, (
                f"request {b}: gpu {emit[b]} oracle {ref.emitted[i]}, "
                f"top-2 gap {gap}")
            ties += 1
    return ref, ties


@pytest.mark.parametrize("B,K,V", [
    (12, 5, 5001),     # one CTA per request, ragged vocabulary
    (40, 3, 4096),     # one CTA per request, float4 loads
    (12, 5, 40000),    # clusters of 8 CTAs
    (12, 4, 40003),    # clusters of 8, ragged slices and a ragged last block
    (1, 1, 9000),      # one request, one draft
    (3, 64, 1024),     # the largest K
    (300, 2, 20000),   # more requests than the GPU has SMs
])
def test_verify_matches_oracle(B, K, V):
    v = wl.make_verify(B, K, V, seed=B * 1000 + K + V)
    acc, emit = _gpu_verify(v)
    ref, ties = _check(v, acc, emit)
    assert ties <= 1
    # the generator's drafts should reach both outcomes on these sizes
    if B >= 12:
        assert (ref.accepted_len < K).any()


def test_verify_branch_cases():
    B, K, V = 16, 4, 40000
    v = wl.make_verify(B, K, V, seed=91)
    rng = np.random.Generator(np.random.PCG64(92))
    for b in range(B):
        d = v.tokens[b]
        if b in (0, 1, 2, 3):
            # every draft accepted (p >= q at every draft) -> bonus draw
            for k in range(K):
                v.p[b, k, d[k]] = 1.0
        if b == 1:
            # bonus row with weights so large e^-best leaves float32's range
            idx = rng.choice(V, size=40, replace=False)
            v.p[b, K, idx] = np.float32(1e36)
        if b == 2:
            # two infinite weights in the bonus row: the lower index wins
            v.p[b, K, [777, 31000]] = np.inf
        if b == 3:
            # an all-zero bonus row: nothing can win, token 0
            v.p[b, K, :] = 0.0
        if b == 4:
            # rejected at 0 with a residual that is zero everywhere: p = q
            # except p[d0] = 0, so the draw falls back to p itself
            v.p[b, 0] = v.q[b, 0]
            v.p[b, 0, d[0]] = 0.0
        if b == 5:
            # rejected at 0 and p_0 all zero: token 0
            v.p[b, 0, :] = 0.0
        if b == 6:
            # NaN probabilities scattered through q and p
            idx = rng.choice(V, size=200, replace=False)
            v.q[b, :, idx[:100]] = np.nan
            v.p[b, :, idx[100:]] = np.nan
        if b == 7:
            # accept 0 and 1 surely, reject at 2 surely (p_2[d] = 0)
            v.p[b, 0, d[0]] = 1.0
            v.p[b, 1, d[1]] = 1.0
            v.p[b, 2, d[2]] = 0.0
        if b == 8:
            # one denormal residual weight, zero elsewhere
            v.p[b, 0] = v.q[b, 0]
            v.p[b, 0, d[0]] = 0.0
            v.q[b, 0, 123] = 0.0
            v.p[b, 0, 123] = np.float32(1e-44)
    acc, emit = _gpu_verify(v)
    ref, ties = _check(v, acc, emit)
    assert ties == 0
    assert list(acc[:4]) == [K] * 4
    assert emit[2] == 777
    assert emit[3] == 0
    assert acc[4] == 0 and acc[5] == 0 and emit[5] == 0
    assert acc[7] == 2
    assert acc[8] == 0 and emit[8] == 123


def test_verify_invalid_draft_marks_only_that_request():
    v = wl.make_verify(6, 3, 9000, seed=5)
    v.tokens[2, 1] = 9000      # out of range
    v.tokens[4, 0] = -1
    acc, emit = _gpu_verify(v)
    assert acc[2] == -1 and emit[2] == -1
    assert acc[4] == -1 and emit[4] == -1
    _check(v, acc, emit, skip=(2, 4))


def test_verify_deterministic_and_offset_sensitive():
    v = wl.make_verify(24, 5, 30000, seed=17)
    a1 = _gpu_verify(v)
    a2 = _gpu_verify(v)
    np.testing.assert_array_equal(a1[0], a2[0])
    np.testing.assert_array_equal(a1[1], a2[1])
    v.offset = v.offset + np.uint64(1)
    a3 = _gpu_verify(v)
    _check(v, *a3)
    assert (a3[1] != a1[1]).any() or (a3[0] != a1[0]).any()


def test_verify_full_size_block():
    # the verification that follows the B=88, K=7, V=200064 draft block
    v = wl.make_verify(88, 7, 200064, seed=1004, logit_std=4.0)
    acc, emit = _gpu_verify(v)
    ref, ties = _check(v, acc, emit)
    assert ties <= 1
    assert 0 < ref.accepted_len.mean() < 7
