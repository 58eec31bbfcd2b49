"""Pins of the fp64 CPU oracle against what the pages and mathematics fix.

Every test here runs on the CPU (no GPU marker).  None of them re-types the
oracle's own formula: each compares the oracle with an independent library
routine (numpy's Philox, torch's log_softmax / argmax, numpy's searchsorted),
with a closed form printed on the pages, with brute-force enumeration, or with
a statistical property (acceptance rate, losslessness) that a dropped term, a
swapped p/q, a wrong row index or a wrong sign would break.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U64 = 2**64 - 1


# --------------------------------------------------------------------------
# Philox-4x64-10 and the uniform draws
# --------------------------------------------------------------------------
def _numpy_block(counter, key):
    """numpy's Philox increments its 256-bit counter before each block, so the
    block for counter c comes from a generator started at c - 1."""
    c = [int(x) for x in counter]
    # subtract one with borrow across the four 64-bit words
    for i in range(4):
        if c[i] > 0:
            c[i] -= 1
            break
        c[i] = U64
    g = np.random.Philox(key=np.array(key, dtype=np.uint64),
                         counter=np.array(c, dtype=np.uint64))
    return g.random_raw(4)


@pytest.mark.parametrize("case", range(12))
def test_philox_matches_numpy(case):
    rng = np.random.default_rng(case)
    counter = rng.integers(0, 2**63, size=4, dtype=np.uint64)
    key = rng.integers(0, 2**63, size=2, dtype=np.uint64)
    if case == 0:
        counter[:] = 0
        key[:] = 0
    if case == 1:
        counter[:] = np.uint64(U64)
        key[:] = np.uint64(U64)
    ours = oracle.philox4x64_10(counter, key)
    assert np.array_equal(ours, _numpy_block(counter, key))


def test_uniform_uses_counter_layout_and_is_odd_multiple():
    key_hi = 0x5350454356455249
    for seed, b, pos, stream in [(0, 0, 0, 0), (7, 3, 2, 1), (2**40 + 5, 255, 7, 0)]:
        u = oracle.uniform(seed, b, pos, stream)
        r0 = int(_numpy_block([b, pos, stream, 0], [seed, key_hi])[0])
        k = u * 2**53
        assert k == int(k) and int(k) % 2 == 1
        assert int(k) // 2 == r0 >> 12
        assert 0.0 < u < 1.0


def test_uniform_has_52_random_bits():
    """u resolves probabilities far below the 2^-23 grid of a float draw: over
    many draws its low bits (below 2^-24) are spread evenly."""
    us = np.array([oracle.uniform(3, b, 1, 1) for b in range(4096)])
    low = np.array([(int(u * 2**53) >> 1) & 0xFFFFFFF for u in us])  # bits 2^-52 .. 2^-25
    assert len(np.unique(low)) > 4000
    assert abs(low.mean() / 2**28 - 0.5) < 0.05


def test_uniform_distribution_ks():
    from scipy import stats
    us = np.array([oracle.uniform(11, b, 0, 0) for b in range(20000)])
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    # streams and positions are different draws
    assert oracle.uniform(11, 0, 0, 0) != oracle.uniform(11, 0, 0, 1)
    assert oracle.uniform(11, 0, 0, 0) != oracle.uniform(11, 0, 1, 0)


# --------------------------------------------------------------------------
# temperature softmax statistics and the gather
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,tau", [(torch.float32, 1.0), (torch.bfloat16, 0.7),
                                       (torch.float32, 2.5)])
def test_row_stats_match_torch_logsumexp(dtype, tau):
    g = torch.Generator().manual_seed(3)
    B, K, V = 3, 3, 257
    target = (4 * torch.randn(B, K + 1, V, generator=g)).to(dtype)
    draft = (4 * torch.randn(B, K, V, generator=g)).to(dtype)
    tokens = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    out = oracle.spec_verify(target, draft, tokens, tau, 5)
    rows = torch.cat([target, draft], dim=1).double() / tau  # (B, 2K+1, V)
    lse = torch.logsumexp(rows, dim=-1).numpy()
    rmax = rows.max(dim=-1).values.numpy()
    np.testing.assert_allclose(out["row_logmax"], rmax, rtol=0, atol=0)
    np.testing.assert_allclose(out["row_logmax"] + np.log(out["row_sum"]), lse,
                               rtol=1e-13, atol=1e-12)
    logp = torch.log_softmax(target.double() / tau, dim=-1)
    logq = torch.log_softmax(draft.double() / tau, dim=-1)
    for b in range(B):
        for i in range(out["n"][b] + 1 if out["n"][b] < K else K):
            x = int(tokens[b, i])
            assert out["px"][b, i] == pytest.approx(math.exp(logp[b, i, x]), rel=1e-12)
            assert out["qx"][b, i] == pytest.approx(math.exp(logq[b, i, x]), rel=1e-12)


def _simple_rows(p_rows, q_rows):
    """fp32 logits whose softmax is (up to fp32 rounding of the logs) the given
    probabilities; zero probabilities become -inf logits.  Returns the logits
    and the exact probabilities those fp32 logits define (torch, fp64)."""
    def logits(P):
        P = np.asarray(P, dtype=np.float64)
        with np.errstate(divide="ignore"):
            return torch.from_numpy(np.log(P).astype(np.float32))
    t = logits(p_rows)
    d = logits(q_rows)
    return t, d, torch.softmax(t.double(), -1).numpy(), torch.softmax(d.double(), -1).numpy()


# --------------------------------------------------------------------------
# acceptance: alpha = E(min(p, q)), q == p, p(x) = 0
# --------------------------------------------------------------------------
def test_acceptance_rate_is_sum_of_min():
    """Page 2, 'How much speedup to expect': alpha = E(min(p, q)).  With x ~ q
    the acceptance frequency at position 0 must equal sum_x min(p(x), q(x))."""
    p0 = [0.5, 0.2, 0.2, 0.1]
    q0 = [0.1, 0.6, 0.2, 0.1]
    t, d, P, Q = _simple_rows([p0, p0], [q0])
    alpha = np.minimum(P[0], Q[0]).sum()
    n_rep = 200000
    rng = np.random.default_rng(1)
    x = rng.choice(4, size=(n_rep, 1), p=Q[0]).astype(np.int32)
    out = oracle.spec_verify(t, d, x, 1.0, 99, broadcast=True, n_seq=n_rep)
    acc = (out["n"] >= 1).mean()
    sigma = math.sqrt(alpha * (1 - alpha) / n_rep)
    assert abs(acc - alpha) < 5 * sigma
    # the swapped ratio q/p would give a different rate here
    swapped = (Q[0] * np.minimum(1, Q[0] / P[0])).sum()
    assert abs(swapped - alpha) > 20 * sigma


def test_identical_draft_accepts_everything():
    """q == p: min(1, p/q) = 1, so every drafted token is kept and the bonus
    token is drawn from p_K."""
    g = torch.Generator().manual_seed(4)
    K, V = 4, 50
    target = 3 * torch.randn(1, K + 1, V, generator=g)
    draft = target[:, :K].clone()
    n_rep = 20000
    x = torch.randint(0, V, (n_rep, K), generator=g, dtype=torch.int32)
    out = oracle.spec_verify(target[0], draft[0], x, 1.0, 3, broadcast=True, n_seq=n_rep)
    assert (out["n"] == K).all()
    assert np.array_equal(out["tokens"][:, :K], x.numpy())


def test_zero_target_probability_always_rejects():
    t, d, P, Q = _simple_rows([[0.0, 0.5, 0.5], [1 / 3] * 3], [[0.5, 0.25, 0.25]])
    x = np.zeros((5000, 1), dtype=np.int32)  # p(0) = 0 < q(0)
    out = oracle.spec_verify(t, d, x, 1.0, 8, broadcast=True, n_seq=5000)
    assert (out["n"] == 0).all()
    # the replacement never lands on a token where p <= q (token 0 here)
    assert (out["tokens"][:, 0] != 0).all()


def test_zero_draft_probability_always_accepts():
    t, d, P, Q = _simple_rows([[0.5, 0.5], [0.5, 0.5]], [[0.0, 1.0]])
    x = np.zeros((1000, 1), dtype=np.int32)  # q(0) = 0 <= p(0)
    out = oracle.spec_verify(t, d, x, 1.0, 8, broadcast=True, n_seq=1000)
    assert (out["n"] == 1).all()


# --------------------------------------------------------------------------
# the residual, the inverse CDF and losslessness
# --------------------------------------------------------------------------
def test_replacement_token_follows_normalised_residual():
    """After a rejection the replacement comes from max(0, p - q) / sum (page 1
    sec. 2, page 2 'The correctness guarantee', page 3 sec. 1)."""
    from scipy import stats
    p0 = [0.05, 0.4, 0.3, 0.05, 0.2]
    q0 = [0.5, 0.1, 0.2, 0.15, 0.05]
    t, d, P, Q = _simple_rows([p0, [0.2] * 5], [q0])
    n_rep = 300000
    x = np.zeros((n_rep, 1), dtype=np.int32)  # p(0)/q(0) = 0.1
    out = oracle.spec_verify(t, d, x, 1.0, 21, broadcast=True, n_seq=n_rep)
    rej = out["n"] == 0
    resid = np.maximum(P[0] - Q[0], 0.0)
    resid /= resid.sum()
    counts = np.bincount(out["tokens"][rej, 0], minlength=5)
    expected = resid * rej.sum()
    mask = expected > 0
    assert counts[~mask].sum() == 0
    assert stats.chisquare(counts[mask], expected[mask]).pvalue > 1e-4
    # resid mass reported by the oracle is sum max(0, p - q)
    np.testing.assert_allclose(out["resid_mass"][rej][:10],
                               np.maximum(P[0] - Q[0], 0).sum(), rtol=1e-12)


def test_inverse_cdf_matches_searchsorted():
    g = torch.Generator().manual_seed(9)
    B, K, V = 64, 3, 300
    target = 2 * torch.randn(B, K + 1, V, generator=g, dtype=torch.float64).float()
    draft = (target[:, :K] + torch.randn(B, K, V, generator=g)).float()
    tokens = torch.multinomial(torch.softmax(draft.reshape(-1, V), -1), 1,
                               generator=g).reshape(B, K).int()
    out = oracle.spec_verify(target, draft, tokens, 1.0, 77)
    P = torch.softmax(target.double(), -1).numpy()
    Q = torch.softmax(draft.double(), -1).numpy()
    checked = 0
    for b in range(B):
        n = out["n"][b]
        r = np.maximum(P[b, n] - Q[b, n], 0) if n < K else P[b, K]
        if out["sample_margin"][b] < 1e-9:
            continue
        j = np.searchsorted(np.cumsum(r), out["theta"][b], side="right")
        assert out["tokens"][b, n] == j
        assert out["theta"][b] == pytest.approx(out["w"][b] * r.sum(), rel=1e-12)
        checked += 1
    assert checked > 50


def _exact_output_marginals(P, Q):
    """Brute force over every drafted tuple x (weight prod q_i(x_i)) and both
    branches of every acceptance test: returns M[j, v] = Pr(position j is
    reached and emits v), from the page formulas alone (min(1, p/q),
    normalised max(0, p - q), bonus p_K)."""
    K = Q.shape[0]
    V = P.shape[1]
    M = np.zeros((K + 1, V))
    for x in itertools.product(range(V), repeat=K):
        w = np.prod([Q[i, x[i]] for i in range(K)])
        if w == 0:
            continue
        reach = w
        for i in range(K):
            a = 1.0 if Q[i, x[i]] == 0 else min(1.0, P[i, x[i]] / Q[i, x[i]])
            resid = np.maximum(P[i] - Q[i], 0)
            if resid.sum() > 0:
                M[i] += reach * (1 - a) * resid / resid.sum()
            M[i, x[i]] += reach * a
            reach *= a
        M[K] += reach * P[K]
    return M


def test_brute_force_enumeration_is_lossless():
    rng = np.random.default_rng(5)
    for K, V in [(1, 3), (2, 3), (3, 4)]:
        P = rng.dirichlet(np.ones(V), size=K + 1)
        Q = rng.dirichlet(np.ones(V), size=K)
        M = _exact_output_marginals(P, Q)
        reach = M.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(M / reach, P, atol=1e-12)


@pytest.mark.parametrize("K,V,seed", [(1, 4, 1), (2, 6, 2), (3, 8, 3)])
def test_chi_square_losslessness(K, V, seed):
    """For every position j, the emitted token given that j was reached follows
    p_j (page 1 sec. 2, page 2 'The correctness guarantee', page 4 sec. 2).
    10^6 replicates, drafts drawn from q with numpy."""
    from scipy import stats
    g = torch.Generator().manual_seed(seed)
    target = (2 * torch.randn(K + 1, V, generator=g)).float()
    draft = (target[:K] + 1.5 * torch.randn(K, V, generator=g)).float()
    P = torch.softmax(target.double(), -1).numpy()
    Q = torch.softmax(draft.double(), -1).numpy()
    n_rep = 1000000
    rng = np.random.default_rng(seed)
    x = np.stack([rng.choice(V, size=n_rep, p=Q[i]) for i in range(K)], axis=1).astype(np.int32)
    out = oracle.spec_verify(target, draft, x, 1.0, 1000 + seed, broadcast=True, n_seq=n_rep)
    M = _exact_output_marginals(P, Q)
    for j in range(K + 1):
        reached = out["n"] >= j
        counts = np.bincount(out["tokens"][reached, j], minlength=V)
        assert stats.chisquare(counts, P[j] * reached.sum()).pvalue > 1e-4
        # how often position j is reached matches the enumeration
        pr = M[j].sum()
        sig = math.sqrt(pr * (1 - pr) / n_rep) + 1e-12
        assert abs(reached.mean() - pr) < 5 * sig


def _adversarial_rows(K, V):
    """Target rows with their mass on the low ids and a draft that puts almost
    all of its mass on the last id, where the target has almost none."""
    target = torch.zeros(K + 1, V)
    target[:, 0], target[:, 1], target[:, V - 1] = 3.0, 2.5, -6.0
    draft = torch.zeros(K, V)
    draft[:, V - 1] = 8.0
    return target, draft


def test_adversarial_draft_is_still_lossless():
    """The output distribution does not depend on how good the draft is
    (page 2 'The correctness guarantee'): a draft concentrated where the
    target is nearly zero is rejected almost always, and the emitted tokens
    still follow p, by exact enumeration and by chi-square over 10^6
    replicas; the acceptance rate is the (small) sum of min(p, q)."""
    from scipy import stats
    K, V, n_rep = 2, 6, 1000000
    target, draft = _adversarial_rows(K, V)
    P = torch.softmax(target.double(), -1).numpy()
    Q = torch.softmax(draft.double(), -1).numpy()
    M = _exact_output_marginals(P, Q)
    np.testing.assert_allclose(M / M.sum(axis=1, keepdims=True), P, atol=1e-12)
    rng = np.random.default_rng(8)
    x = np.stack([rng.choice(V, size=n_rep, p=Q[i]) for i in range(K)], axis=1).astype(np.int32)
    out = oracle.spec_verify(target, draft, x, 1.0, 77, broadcast=True, n_seq=n_rep)
    alpha = np.minimum(P[0], Q[0]).sum()
    assert alpha < 0.05
    acc0 = (out["n"] >= 1).mean()
    assert abs(acc0 - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / n_rep)
    for j in range(K + 1):
        reached = out["n"] >= j
        counts = np.bincount(out["tokens"][reached, j], minlength=V)
        assert stats.chisquare(counts, P[j] * reached.sum()).pvalue > 1e-4


def test_expected_tokens_closed_form_and_page_example():
    """Page 2: E[tokens] = (1 - alpha^(gamma+1)) / (1 - alpha); worked example
    0.7 -> about 2.8, 0.9 -> about 4.1 for gamma = 4 (tests/golden)."""
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "expected_tokens.txt"))
            if ln.strip() and not ln.startswith("#")]
    for a_s, g_s, printed in rows:
        alpha, gamma = float(a_s), int(g_s)
        closed = (1 - alpha ** (gamma + 1)) / (1 - alpha)
        assert abs(closed - float(printed)) <= 0.05
        # rows with a fixed per-position acceptance alpha: q = (1, 0),
        # p = (alpha, 1 - alpha), so x = 0 is accepted with probability alpha
        t, d, P, Q = _simple_rows([[alpha, 1 - alpha]] * (gamma + 1), [[1.0, 0.0]] * gamma)
        a = P[0, 0]
        n_rep = 400000
        x = np.zeros((n_rep, gamma), dtype=np.int32)
        out = oracle.spec_verify(t, d, x, 1.0, 31, broadcast=True, n_seq=n_rep)
        tokens_per_iter = out["n"] + 1
        mean = tokens_per_iter.mean()
        expect = (1 - a ** (gamma + 1)) / (1 - a)
        assert abs(mean - expect) < 5 * tokens_per_iter.std() / math.sqrt(n_rep)


# --------------------------------------------------------------------------
# temperature, greedy, bad data
# --------------------------------------------------------------------------
def test_temperature_divides_both_models():
    """Scaling logits and temperature together changes nothing."""
    g = torch.Generator().manual_seed(12)
    B, K, V = 8, 3, 64
    target = torch.randn(B, K + 1, V, generator=g)
    draft = torch.randn(B, K, V, generator=g)
    tokens = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    a = oracle.spec_verify(target, draft, tokens, 0.5, 4)
    b = oracle.spec_verify(target * 4, draft * 4, tokens, 2.0, 4)
    assert np.array_equal(a["tokens"], b["tokens"]) and np.array_equal(a["n"], b["n"])
    np.testing.assert_allclose(a["px"], b["px"], rtol=1e-6, equal_nan=True)


def test_greedy_matches_torch_argmax():
    g = torch.Generator().manual_seed(2)
    B, K, V = 40, 4, 1000
    target = (4 * torch.randn(B, K + 1, V, generator=g)).to(torch.bfloat16)
    # plant exact ties: copy the max value to a later and an earlier index
    target[0, 0, 10] = 30.0
    target[0, 0, 900] = 30.0
    amax = torch.argmax(target.float(), dim=-1).int()
    tokens = amax[:, :K].clone()
    tokens[::3, 2] = (tokens[::3, 2] + 1) % V
    out = oracle.spec_verify_greedy(target, tokens)
    assert np.array_equal(out["row_argmax"], amax.numpy())
    assert out["row_argmax"][0, 0] == 10
    for b in range(B):
        n = 2 if b % 3 == 0 else K
        assert out["n"][b] == n
        assert list(out["tokens"][b, :n]) == list(tokens[b, :n].numpy())
        assert out["tokens"][b, n] == amax[b, n]
        assert (out["tokens"][b, n + 1:] == -1).all()


def test_bad_data_marks_sequence():
    g = torch.Generator().manual_seed(6)
    B, K, V = 5, 2, 16
    target = torch.randn(B, K + 1, V, generator=g)
    draft = torch.randn(B, K, V, generator=g)
    tokens = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    target[1, 2, 3] = float("nan")
    draft[2, 0, :] = float("-inf")
    tokens[3, 1] = V
    target[4, 0, 5] = float("inf")
    out = oracle.spec_verify(target, draft, tokens, 1.0, 1)
    assert list(out["n"]) [1:] == [-1, -1, -1, -1]
    assert out["n"][0] >= 0
    assert (out["tokens"][1:] == -1).all()
    # -inf entries alone are legal (masked vocabulary)
    target2 = target[:1].clone()
    target2[0, :, 7] = float("-inf")
    assert oracle.spec_verify(target2, draft[:1], tokens[:1], 1.0, 1)["n"][0] >= 0


# --------------------------------------------------------------------------
# tree verification
# --------------------------------------------------------------------------
def _ancestors_closed_form(i, j):
    """Complete binary tree in BFS order with the root outside the node list:
    node j is an ancestor-or-self of node i iff (j + 2) == (i + 2) >> k, k >= 0."""
    a, b = i + 2, j + 2
    while a >= b:
        if a == b:
            return True
        a >>= 1
    return False


def test_tree_mask_closed_form_and_brute_force():
    from speculative_decoding_verification_36_gb300.workloads import complete_binary_parents
    depth = 4
    par = complete_binary_parents(depth).numpy()
    N = len(par)
    assert N == 30
    V = 8
    target = torch.zeros(1, N + 1, V)
    out = oracle.tree_verify_greedy(target, np.zeros((1, N), np.int32), par[None])
    mask = out["mask"][0, :, 0]
    for i in range(N):
        for j in range(N):
            bit = (int(mask[i]) >> j) & 1
            assert bit == int(_ancestors_closed_form(i, j))


def _paths_brute_force(par):
    """All root-to-node paths, as node lists."""
    paths = []
    for i in range(len(par)):
        p, node = [], i
        while node != -1:
            p.append(node)
            node = par[node]
        paths.append(p[::-1])
    return paths


@pytest.mark.parametrize("seed", range(6))
def test_tree_path_brute_force(seed):
    rng = np.random.default_rng(seed)
    N, V = 25, 6
    par = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, N)], dtype=np.int32)
    target = torch.from_numpy(rng.normal(size=(2, N + 1, V)).astype(np.float32))
    g = torch.argmax(target, -1).numpy()
    tok = rng.integers(0, V, size=(2, N)).astype(np.int32)
    # make roughly half the nodes match their parent's argmax
    for b in range(2):
        for i in range(N):
            if rng.random() < 0.6:
                tok[b, i] = g[b, par[i] + 1]
    out = oracle.tree_verify_greedy(target, tok, np.stack([par, par]))
    for b in range(2):
        best = []
        for p in _paths_brute_force(par):
            if all(tok[b, node] == g[b, par[node] + 1] for node in p) and len(p) > len(best):
                best = p
        exp = [int(tok[b, node]) for node in best] + [int(g[b, (best[-1] + 1) if best else 0])]
        assert out["length"][b] == len(exp)
        assert list(out["path"][b, :len(exp)]) == exp
        assert (out["path"][b, len(exp):] == -1).all()
        # mask rows: ancestor-or-self from the explicit path lists
        for i, p in enumerate(_paths_brute_force(par)):
            words = out["mask"][b, i]
            got = {j for j in range(N) if (int(words[j // 32]) >> (j % 32)) & 1}
            assert got == set(p)


def test_tree_bad_parent_is_flagged():
    target = torch.zeros(1, 4, 5)
    out = oracle.tree_verify_greedy(target, np.zeros((1, 3), np.int32),
                                    np.array([[-1, 0, 2]], np.int32))
    assert out["length"][0] == -1 and (out["path"] == -1).all() and (out["mask"] == 0).all()


# --------------------------------------------------------------------------
# acceptance statistics (page 2, "How much speedup to expect")
# --------------------------------------------------------------------------
def test_acceptance_stats_worked_example():
    """Counted by hand: n = 0, 1, 2, 4, 4, bad, 3, 0 with K = 4."""
    r = oracle.acceptance_stats([0, 1, 2, 4, 4, -1, 3, 0], 4)
    assert r["hist"].tolist() == [2, 1, 1, 1, 2, 1]
    # position i tested by #(n >= i) sequences, accepted by #(n > i)
    assert np.allclose(r["alpha"], [5 / 7, 4 / 5, 3 / 4, 2 / 3], rtol=0, atol=1e-15)
    assert r["mean_tokens"] == (2 * 1 + 1 * 2 + 1 * 3 + 1 * 4 + 2 * 5) / 7


def test_acceptance_stats_edge_cases():
    empty = oracle.acceptance_stats([], 3)
    assert empty["hist"].tolist() == [0, 0, 0, 0, 0]
    assert np.isnan(empty["alpha"]).all() and math.isnan(empty["mean_tokens"])
    bad = oracle.acceptance_stats([-1, 7, -5], 3)  # every value outside [0, K]
    assert bad["hist"].tolist() == [0, 0, 0, 0, 3] and math.isnan(bad["mean_tokens"])
    none = oracle.acceptance_stats([0, 0, 2], 0)  # K = 0: only n == 0 counts
    assert none["hist"].tolist() == [2, 1] and none["alpha"].size == 0
    assert none["mean_tokens"] == 1.0


@pytest.mark.parametrize("alpha", [0.7, 0.9])
def test_acceptance_stats_recover_alpha_and_closed_form(alpha):
    """Positions accepted independently with probability alpha: the histogram is
    numpy.bincount, every alpha_i estimates alpha, and the mean tokens per
    iteration approaches the page's (1 - alpha^(K+1)) / (1 - alpha)."""
    K, B = 4, 400000
    rng = np.random.default_rng(5)
    acc = rng.random((B, K)) < alpha
    n = np.where(acc.all(axis=1), K, np.argmin(acc, axis=1)).astype(np.int32)
    r = oracle.acceptance_stats(n, K)
    assert r["hist"][:K + 1].tolist() == np.bincount(n, minlength=K + 1).tolist()
    assert r["hist"][K + 1] == 0
    for i in range(K):
        reached = int((n >= i).sum())
        assert abs(r["alpha"][i] - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / reached)
    expect = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(r["mean_tokens"] - expect) < 5 * (n + 1).std() / math.sqrt(B)


# --------------------------------------------------------------------------
# per-row entropy (page 3, sec. 3: speculation depth from the distribution's
# uncertainty)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("tau", [0.5, 1.0, 1.7])
def test_row_entropy_matches_torch_categorical(dtype, tau):
    g = torch.Generator().manual_seed(31)
    z = (torch.randn(4, 3, 513, generator=g) * 3).to(dtype)
    h = oracle.row_entropy(z, tau)
    ref = torch.distributions.Categorical(logits=z.double() / tau).entropy().numpy()
    assert np.abs(h - ref).max() < 1e-12


def test_row_entropy_closed_forms():
    V = 1000
    assert abs(oracle.row_entropy(torch.zeros(1, V), 1.0)[0] - math.log(V)) < 1e-12  # uniform
    one_hot = torch.full((1, V), -float("inf"))
    one_hot[0, 17] = 3.0
    assert oracle.row_entropy(one_hot, 0.9)[0] == 0.0
    two = torch.full((1, V), -float("inf"))  # two admissible tokens
    two[0, 0], two[0, 1] = math.log(0.3), math.log(0.7)
    l0, l1 = float(two[0, 0]), float(two[0, 1])  # the fp32-rounded logits
    a = 1.0 / (1.0 + math.exp(l1 - l0))
    expect = -a * math.log(a) - (1 - a) * math.log(1 - a)
    assert abs(oracle.row_entropy(two, 1.0)[0] - expect) < 1e-12
    bad = torch.zeros(2, 8)
    bad[0, 3] = float("nan")
    bad[1, :] = -float("inf")
    assert np.isnan(oracle.row_entropy(bad, 1.0)).all()


# --------------------------------------------------------------------------
# adaptive draft length (page 3, sec. 3 "Engineering Recommendations")
# --------------------------------------------------------------------------
def _khint_batch(tau=0.7):
    """Four sequences, K = 3, V = 64, whose target row i is uniform over its
    first M_i tokens (entropy ln M_i exactly), M = (8, 1, 64, 2):
      0: drafts equal to the target rows, tokens inside the support: n = 3;
      1: draft row 0 uniform over 32 tokens, token 10 has p = 0: n = 0;
      2: position 0 drafted from the target row itself (accepted), token 5 at
         position 1 has p = 0: n = 1;
      3: a NaN logit in target row 2: bad."""
    K, V = 3, 64
    M = (8, 1, 64, 2)
    target = torch.full((4, K + 1, V), -float("inf"))
    for i, m in enumerate(M):
        target[:, i, :m] = 0.0
    draft = target[:, :K].clone()
    tokens = torch.zeros(4, K, dtype=torch.int32)
    draft[1, 0] = -float("inf")
    draft[1, 0, :32] = 0.0
    tokens[1, 0] = 10
    tokens[2, 0] = 3
    tokens[2, 1] = 5
    draft[2, 1] = 0.0  # uniform over all 64: q(5) > 0 = p(5)
    target[3, 2, 7] = float("nan")
    return target, draft, tokens, K, M, tau


def test_adaptive_k_closed_forms():
    target, draft, tokens, K, M, tau = _khint_batch()
    out = oracle.spec_verify(target, draft, tokens, tau, 5)
    assert out["n"].tolist() == [3, 0, 1, -1]
    h = oracle.row_entropy(target, tau)
    ln = [math.log(m) for m in M]
    assert np.abs(h[:3] - np.array(ln)).max() < 1e-12
    r = oracle.adaptive_k(h, out["n"], K, 1.2, 1.9, 1, 8)
    # mean over target rows 0..n: 2.5 ln 2, ln 8, 1.5 ln 2
    want = [2.5 * math.log(2), 3 * math.log(2), 1.5 * math.log(2)]
    assert np.abs(r["mean_entropy"][:3] - np.array(want)).max() < 1e-12
    assert np.isnan(r["mean_entropy"][3])
    # 1.73 in [1.2, 1.9]: keep; 2.08 > 1.9: lower; 1.04 < 1.2: raise; bad: -1
    assert r["k_next"].tolist() == [3, 2, 4, -1]


def test_adaptive_k_clamps_and_bounds():
    target, draft, tokens, K, M, tau = _khint_batch()
    out = oracle.spec_verify(target, draft, tokens, tau, 5)
    h = oracle.row_entropy(target, tau)
    assert oracle.adaptive_k(h, out["n"], K, 1.2, 1.9, 3, 3)["k_next"].tolist() == [3, 3, 3, -1]
    assert oracle.adaptive_k(h, out["n"], K, 1.2, 1.9, 0, 2)["k_next"].tolist() == [2, 2, 2, -1]
    assert oracle.adaptive_k(h, out["n"], K, 1.2, 1.9, 5, 9)["k_next"].tolist() == [5, 5, 5, -1]
    # every mean below h_lo: all raised; every mean above h_hi: all lowered
    assert oracle.adaptive_k(h, out["n"], K, 10.0, 10.0, 0, 255)["k_next"].tolist() == [4, 4, 4, -1]
    assert oracle.adaptive_k(h, out["n"], K, -1.0, -1.0, 0, 255)["k_next"].tolist() == [2, 2, 2, -1]
    # K = 0: only the bonus row counts
    h0 = np.array([[0.5], [3.0]])
    assert oracle.adaptive_k(h0, [0, 0], 0, 1.0, 2.0, 0, 4)["k_next"].tolist() == [1, 0]
    with pytest.raises(ValueError):
        oracle.adaptive_k(h, out["n"], K, 2.0, 1.0, 0, 8)
    with pytest.raises(ValueError):
        oracle.adaptive_k(h, out["n"], K, 1.0, 2.0, 5, 4)


# --------------------------------------------------------------------------
# stochastic tree verification (page 4, sec. 4, with the page 1 sec. 2 rule)
# --------------------------------------------------------------------------
def test_tree_sampling_on_a_chain_is_the_chain_verify():
    """A tree whose nodes form one chain is verified exactly like the chain."""
    g = torch.Generator().manual_seed(3)
    B, K, V = 64, 5, 50
    T = torch.randn(B, K + 1, V, generator=g) * 2
    D = T + torch.randn(B, K + 1, V, generator=g)
    x = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    par = torch.arange(-1, K - 1, dtype=torch.int32).expand(B, K).contiguous()
    tr = oracle.tree_verify_sampling(T, D, x, par, 0.8, 5)
    ch = oracle.spec_verify(T, D[:, :K].contiguous(), x, 0.8, 5)
    assert np.array_equal(tr["length"], ch["n"] + 1)
    assert np.array_equal(tr["path"], ch["tokens"])


def test_tree_sampling_without_nodes_draws_the_bonus():
    g = torch.Generator().manual_seed(4)
    T = torch.randn(32, 1, 40, generator=g)
    D = torch.randn(32, 1, 40, generator=g)
    tr = oracle.tree_verify_sampling(T, D, torch.zeros(32, 0, dtype=torch.int32),
                                     torch.zeros(32, 0, dtype=torch.int32), 1.3, 8)
    ch = oracle.spec_verify(T, torch.zeros(32, 0, 40), torch.zeros(32, 0, dtype=torch.int32), 1.3, 8)
    assert (tr["length"] == 1).all() and np.array_equal(tr["path"][:, 0], ch["tokens"][:, 0])


def test_tree_sampling_is_lossless():
    """Root with two children drawn from Q_root, each with one child drawn from
    Q1[token].  Target rows depend only on the token prefix, so every emitted
    position, given its prefix and that it exists, must follow the target's
    conditional distribution, whichever sibling was accepted or resampled."""
    from scipy import stats
    V, B = 4, 200000
    rng = np.random.default_rng(11)

    def dist(k):
        p = rng.random(k) + 0.05
        return p / p.sum()
    P0, Q0 = dist(V), dist(V)
    P1 = np.stack([dist(V) for _ in range(V)])
    Q1 = np.stack([dist(V) for _ in range(V)])
    P2 = np.stack([[dist(V) for _ in range(V)] for _ in range(V)])
    c = np.stack([rng.choice(V, size=B, p=Q0), rng.choice(V, size=B, p=Q0)], axis=1)
    gch = np.stack([np.array([rng.choice(V, p=Q1[a]) for a in col]) for col in c.T], axis=1)
    tokens = np.concatenate([c, gch], axis=1).astype(np.int32)
    parents = np.tile(np.array([-1, -1, 0, 1], dtype=np.int32), (B, 1))
    lg = lambda p: np.log(p).astype(np.float32)
    T = np.empty((B, 5, V), dtype=np.float32)
    D = np.empty((B, 5, V), dtype=np.float32)
    T[:, 0] = lg(P0)
    D[:, 0] = lg(Q0)
    for k in range(2):
        T[:, 1 + k] = lg(P1[c[:, k]])
        D[:, 1 + k] = lg(Q1[c[:, k]])
        T[:, 3 + k] = lg(P2[c[:, k], gch[:, k]])
        D[:, 3 + k] = lg(np.full(V, 1.0 / V))  # leaves: their Q is never used
    out = oracle.tree_verify_sampling(T, D, tokens, parents, 1.0, 21)
    path, length = out["path"], out["length"]
    assert length.min() >= 1 and length.max() <= 3
    P0e = np.exp(T[0, 0].astype(np.float64)); P0e /= P0e.sum()
    assert stats.chisquare(np.bincount(path[:, 0], minlength=V), P0e * B).pvalue > 1e-3
    for a in range(V):
        sel = (length >= 2) & (path[:, 0] == a)
        if sel.sum() > 500:
            p = np.exp(lg(P1[a]).astype(np.float64)); p /= p.sum()
            assert stats.chisquare(np.bincount(path[sel, 1], minlength=V), p * sel.sum()).pvalue > 1e-3
        for b2 in range(V):
            sel3 = (length == 3) & (path[:, 0] == a) & (path[:, 1] == b2)
            if sel3.sum() > 500:
                p = np.exp(lg(P2[a, b2]).astype(np.float64)); p /= p.sum()
                assert stats.chisquare(np.bincount(path[sel3, 2], minlength=V),
                                       p * sel3.sum()).pvalue > 1e-3
    # the second sibling is really tested (after a residual update)
    first_rejected = path[:, 0] != c[:, 0]
    assert ((length >= 2) & first_rejected & (path[:, 0] == c[:, 1])).sum() > 1000


def test_tree_sampling_bad_data():
    T = torch.zeros(3, 3, 8)
    D = torch.zeros(3, 3, 8)
    tok = torch.tensor([[1, 2], [1, 9], [1, 2]], dtype=torch.int32)  # sequence 1: token out of range
    par = torch.tensor([[-1, 0], [-1, 0], [-1, 1]], dtype=torch.int32)  # sequence 2: parent not < i
    out = oracle.tree_verify_sampling(T, D, tok, par, 1.0, 0)
    assert out["length"].tolist()[1:] == [-1, -1] and (out["path"][1:] == -1).all()
    assert out["length"][0] >= 1


# --------------------------------------------------------------------------
# n-gram (prompt-lookup) drafting
# --------------------------------------------------------------------------
def _ngram_by_index(h, n_min, n_max, K):
    """The same reading by a different route: for each match length m a
    dictionary from every m-gram of the history to the end (exclusive) of its
    latest occurrence that still has a following token, then one lookup of
    the last m tokens."""
    L = len(h)
    for m in range(n_max, n_min - 1, -1):
        if L < m + 1:
            continue
        last_end = {}
        for e in range(m, L):  # e <= L - 1: one token follows
            last_end[tuple(h[e - m:e])] = e
        e = last_end.get(tuple(h[L - m:L]))
        if e is not None:
            d = min(K, L - e)
            return list(h[e:e + d]), d, m
    return [], 0, 0


def test_ngram_worked_cases():
    cases = [
        # suffix (5,6,7) also ends at 3; the three tokens after it are 8,5,6
        ([5, 6, 7, 8, 5, 6, 7], 2, 3, 3, [8, 5, 6], 3),
        # a run: the latest earlier (9,9) ends at 3, one token (9) follows
        ([9, 9, 9, 9], 1, 2, 4, [9], 2),
        # (9,3,4) never occurred before; (3,4) ends at 4; drafts 9,3,4
        ([1, 2, 3, 4, 9, 3, 4], 1, 3, 3, [9, 3, 4], 2),
        # two earlier (1,2): the latest one (end 5) wins, then 7 and the 1,2
        ([1, 2, 3, 1, 2, 7, 1, 2], 2, 2, 4, [7, 1, 2], 2),
        # nothing repeats
        ([1, 2, 3, 4, 5], 1, 3, 2, [], 0),
        # K = 0: a match, no drafts
        ([4, 4, 4], 1, 1, 0, [], 1),
    ]
    for h, n_min, n_max, K, want, m in cases:
        out = oracle.ngram_draft(np.array([h], dtype=np.int32), [len(h)], n_min, n_max, K)
        d = int(out["n_drafts"][0])
        assert d == len(want) and out["drafts"][0, :d].tolist() == want, (h, out)
        assert (out["drafts"][0, d:] == -1).all()
        assert int(out["match_len"][0]) == m, (h, out)


def test_ngram_matches_the_dictionary_index():
    rng = np.random.default_rng(7)
    for trial in range(400):
        B = int(rng.integers(1, 6))
        Lmax = int(rng.integers(1, 60))
        alphabet = int(rng.integers(2, 6))
        toks = rng.integers(0, alphabet, size=(B, Lmax)).astype(np.int32)
        lengths = rng.integers(0, Lmax + 1, size=B).astype(np.int32)
        n_min = int(rng.integers(1, 4))
        n_max = n_min + int(rng.integers(0, 4))
        K = int(rng.integers(0, 7))
        out = oracle.ngram_draft(toks, lengths, n_min, n_max, K)
        for b in range(B):
            want, d, m = _ngram_by_index(toks[b, :lengths[b]].tolist(), n_min, n_max, K)
            assert int(out["n_drafts"][b]) == d and int(out["match_len"][b]) == m
            assert out["drafts"][b, :d].tolist() == want
            assert (out["drafts"][b, d:] == -1).all()


def test_ngram_copy_property_and_bad_lengths():
    rng = np.random.default_rng(11)
    toks = rng.integers(0, 3, size=(8, 200)).astype(np.int32)
    lengths = np.array([200, 150, 3, 2, 1, 0, -1, 201], dtype=np.int32)
    out = oracle.ngram_draft(toks, lengths, 2, 5, 6)
    for b in range(6):
        L, m, d = int(lengths[b]), int(out["match_len"][b]), int(out["n_drafts"][b])
        if m == 0:
            assert d == 0
            continue
        h = toks[b, :L]
        # the drafts continue an earlier copy of the last m tokens
        e = next(e for e in range(L - 1, m - 1, -1)
                 if (h[e - m:e] == h[L - m:L]).all() and (h[e:e + d] == out["drafts"][b, :d]).all())
        assert d == min(6, L - e)
        # no longer match exists anywhere earlier
        if m < 5:
            mm = m + 1
            assert not any((h[e2 - mm:e2] == h[L - mm:L]).all() for e2 in range(mm, L)) or L < mm + 1
    for b in (6, 7):
        assert out["n_drafts"][b] == -1 and out["match_len"][b] == -1 and (out["drafts"][b] == -1).all()


# --------------------------------------------------------------------------
# the early-exit reading of the bad-data rule
# --------------------------------------------------------------------------
def test_used_rows_only_agrees_on_clean_data_and_ignores_rows_after_n():
    rng = np.random.default_rng(21)
    B, K, V = 40, 5, 64
    t = torch.tensor(2.0 * rng.standard_normal((B, K + 1, V)), dtype=torch.float32)
    d = t[:, :K] + torch.tensor(1.5 * rng.standard_normal((B, K, V)), dtype=torch.float32)
    x = torch.tensor(rng.integers(0, V, (B, K)), dtype=torch.int32)
    full = oracle.spec_verify(t, d, x, 1.0, 9)
    used = oracle.spec_verify(t, d, x, 1.0, 9, used_rows_only=True)
    assert np.array_equal(full["tokens"], used["tokens"]) and np.array_equal(full["n"], used["n"])
    # spoil every row and token after each sequence's first rejection: the
    # used-rows result must not move, while the full rule flags the sequence
    t2, d2, x2 = t.clone(), d.clone(), x.clone()
    spoiled = []
    for b in range(B):
        n = int(full["n"][b])
        if n < K - 1:
            t2[b, n + 1, 3] = float("nan")
            d2[b, K - 1, :] = float("-inf")
            x2[b, K - 1] = V + 5
            spoiled.append(b)
        if n < K:
            t2[b, K, 0] = float("inf")  # the bonus row is not used after a rejection
    assert spoiled
    used2 = oracle.spec_verify(t2, d2, x2, 1.0, 9, used_rows_only=True)
    assert np.array_equal(used2["tokens"], full["tokens"]) and np.array_equal(used2["n"], full["n"])
    full2 = oracle.spec_verify(t2, d2, x2, 1.0, 9)
    assert (full2["n"][spoiled] == -1).all()


def test_used_rows_only_flags_bad_rows_it_uses():
    B, K, V = 4, 3, 16
    t = torch.zeros(B, K + 1, V)
    d = torch.zeros(B, K, V)
    x = torch.zeros(B, K, dtype=torch.int32)  # q = p: every draft accepted
    t[0, 0, 2] = float("nan")       # position 0
    d[1, 2, :] = float("-inf")      # position 2 (reached: all accepted)
    x[2, 1] = -3                     # position 1
    t[3, K, 4] = float("nan")       # the bonus row, used since all are accepted
    out = oracle.spec_verify(t, d, x, 1.0, 0, used_rows_only=True)
    assert out["n"].tolist() == [-1, -1, -1, -1] and (out["tokens"] == -1).all()


def test_greedy_used_rows_only():
    """The early-exit reading of the greedy verify: on clean data the result
    equals the full greedy verify (argmax of torch, lowest id on ties); rows
    and tokens after the first mismatch never matter; a bad row or token at
    or before it marks the sequence bad, and target row K matters only when
    every draft matches."""
    rng = np.random.default_rng(31)
    B, K, V = 60, 4, 32
    t = torch.tensor(2.0 * rng.standard_normal((B, K + 1, V)), dtype=torch.float32)
    g = torch.argmax(t, dim=-1).numpy()
    # drafts match the argmax with probability 0.6 per position
    x = np.where(rng.random((B, K)) < 0.6, g[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    full = oracle.spec_verify_greedy(t, x)
    used = oracle.spec_verify_greedy(t, x, used_rows_only=True)
    assert np.array_equal(full["tokens"], used["tokens"]) and np.array_equal(full["n"], used["n"])
    for b in range(B):
        n = int(used["n"][b])
        assert np.array_equal(used["row_argmax"][b, :n + 1], g[b, :n + 1])
        assert (used["row_argmax"][b, n + 1:] == -1).all()
    assert (full["n"] < K).any() and (full["n"] == K).any()
    # spoil every row and token after each sequence's first mismatch
    t2, x2 = t.clone(), x.copy()
    for b in range(B):
        n = int(full["n"][b])
        if n < K:
            t2[b, n + 1:, 5] = float("nan")
            x2[b, n + 1:] = V + 7
    used2 = oracle.spec_verify_greedy(t2, x2, used_rows_only=True)
    assert np.array_equal(used2["tokens"], used["tokens"]) and np.array_equal(used2["n"], used["n"])
    full2 = oracle.spec_verify_greedy(t2, x2)
    assert all(full2["n"][b] == -1 for b in range(B) if full["n"][b] < K - 1)
    # a bad row at or before n, or an out-of-range x_n, marks the sequence bad
    for b in range(B):
        n = int(full["n"][b])
        t3, x3 = t.clone(), x.copy()
        j = int(rng.integers(0, n + 1))
        t3[b, j, 0] = float("inf")
        assert oracle.spec_verify_greedy(t3, x3, used_rows_only=True)["n"][b] == -1
        if n < K:
            x3 = x.copy()
            x3[b, n] = -5
            r = oracle.spec_verify_greedy(t, x3, used_rows_only=True)
            assert r["n"][b] == -1 and (r["tokens"][b] == -1).all()
    # target row K is used only when every draft matches
    allm = [b for b in range(B) if full["n"][b] == K]
    some = [b for b in range(B) if full["n"][b] < K]
    t4 = t.clone()
    t4[:, K, :] = float("-inf")
    r = oracle.spec_verify_greedy(t4, x, used_rows_only=True)
    assert all(r["n"][b] == -1 for b in allm)
    assert all(r["n"][b] == full["n"][b] for b in some)


def test_tree_used_rows_only():
    """The early-exit reading of the greedy tree verify: on clean data it
    equals the full verify (pinned above by brute force); rows and tokens
    under a rejected node never matter; a bad row of an accepted node (or of
    the root), a bad token under an accepted parent, or a bad parent index
    anywhere marks the sequence bad."""
    rng = np.random.default_rng(41)
    B, V = 48, 24
    par = [-1, -1, 0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5]  # depth-3 binary tree
    N = len(par)
    t = torch.tensor(2.0 * rng.standard_normal((B, N + 1, V)), dtype=torch.float32)
    g = torch.argmax(t, dim=-1).numpy()
    tok = np.zeros((B, N), dtype=np.int32)
    for i, p in enumerate(par):  # a node carries its parent's argmax with probability 0.6
        tok[:, i] = np.where(rng.random(B) < 0.6, g[:, p + 1], rng.integers(0, V, B))
    parents = np.tile(np.array(par, dtype=np.int32), (B, 1))
    full = oracle.tree_verify_greedy(t, tok, parents)
    used = oracle.tree_verify_greedy(t, tok, parents, used_rows_only=True)
    for k in ("path", "length", "mask"):
        assert np.array_equal(full[k], used[k])
    assert len(set(full["length"].tolist())) > 1

    def accepted(b):
        acc = []
        for i, p in enumerate(par):
            acc.append((p < 0 or acc[p]) and tok[b, i] == g[b, p + 1])
        return acc

    # spoil the rows and tokens of every node under a rejected node
    t2, tok2 = t.clone(), tok.copy()
    for b in range(B):
        acc = accepted(b)
        for i, p in enumerate(par):
            if p >= 0 and not acc[p]:
                t2[b, i + 1, 0] = float("nan")
                tok2[b, i] = V + 3
            if not acc[i]:
                t2[b, i + 1, 1] = float("inf")  # a rejected node's own row is unused too
    used2 = oracle.tree_verify_greedy(t2, tok2, parents, used_rows_only=True)
    for k in ("path", "length", "mask"):
        assert np.array_equal(used2[k], used[k])
    assert (oracle.tree_verify_greedy(t2, tok2, parents)["length"] == -1).any()
    # used rows and tokens are checked
    for b in range(0, B, 5):
        acc = accepted(b)
        t3 = t.clone()
        t3[b, 0, 2] = float("nan")
        assert oracle.tree_verify_greedy(t3, tok, parents, used_rows_only=True)["length"][b] == -1
        ai = [i for i in range(N) if acc[i]]
        if ai:
            t3 = t.clone()
            t3[b, ai[-1] + 1, :] = float("-inf")
            assert oracle.tree_verify_greedy(t3, tok, parents, used_rows_only=True)["length"][b] == -1
        tok3 = tok.copy()
        tok3[b, 0] = -1  # node 0's parent is the root, always accepted
        assert oracle.tree_verify_greedy(t, tok3, parents, used_rows_only=True)["length"][b] == -1
        par3 = parents.copy()
        par3[b, N - 1] = N  # a bad parent index anywhere
        assert oracle.tree_verify_greedy(t, tok, par3, used_rows_only=True)["length"][b] == -1
