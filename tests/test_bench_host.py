"""Host logic of bench.py that needs no GPU: the parity check of the bench
line against the oracle, the algorithmic byte count and the stored traffic
figure's source guard."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
import bench  # noqa: E402
import oracle  # noqa: E402
from speculative_decoding_verification_36_gb300 import workloads as wl  # noqa: E402


@pytest.fixture(scope="module")
def first():
    p = wl.preset("c3", B=12, V=4096)
    x = wl.make_chain(p, seed=3)
    return p, {b: oracle.spec_verify(x["target"][b:b + 1], x["draft"][b:b + 1], x["tokens"][b:b + 1],
                                     p.temperature, 0, seq_ids=[b]) for b in range(p.B)}


def _gpu_like(first):
    tok = np.stack([first[b]["tokens"][0] for b in sorted(first)])
    n = np.array([first[b]["n"][0] for b in sorted(first)], dtype=np.int32)
    return tok.copy(), n.copy()


def test_parity_sample_counts_identical_results(first):
    p, ref = first
    tok, n = _gpu_like(ref)
    r = bench.parity_sample(tok, n, ref)
    assert r == {"sequences": p.B, "identical": p.B, "boundary_only": 0, "mismatch": 0,
                 "oracle_boundary_draws": r["oracle_boundary_draws"]}


def test_parity_sample_flags_a_changed_token_or_count(first):
    p, ref = first
    tok, n = _gpu_like(ref)
    b = 2
    tok[b, n[b]] = (tok[b, n[b]] + 1) % p.V  # a different emitted token, far from any boundary
    r = bench.parity_sample(tok, n, ref)
    assert r["mismatch"] == 1 and r["identical"] == p.B - 1
    tok, n = _gpu_like(ref)
    n[5] = -1  # a sequence flagged bad on one side only
    assert bench.parity_sample(tok, n, ref)["mismatch"] == 1


def test_parity_sample_accepts_a_difference_at_a_boundary_draw(first):
    p, ref = first
    tok, n = _gpu_like(ref)
    b = 4
    ref = dict(ref)
    r4 = dict(ref[b])
    # pretend the oracle's acceptance draw at the first rejection sat on the boundary
    am = r4["acc_margin"].copy()
    nb = int(r4["n"][0])
    if nb >= p.K:
        pytest.skip("sequence accepted every draft")
    am[0, nb] = 1e-9
    r4["acc_margin"] = am
    ref[b] = r4
    n[b] = nb + 1  # the GPU accepted the boundary draw
    r = bench.parity_sample(tok, n, ref)
    assert r["boundary_only"] == 1 and r["mismatch"] == 0 and r["oracle_boundary_draws"] >= 1


def test_algorithmic_bytes_of_c3():
    p = wl.preset("c3")
    # 17 rows of 152064 bf16 per sequence, plus drafted tokens and outputs
    assert bench.algorithmic_bytes(p) == 256 * 17 * 152064 * 2 + 256 * 8 * 4 + 256 * 10 * 4


def test_stored_traffic_is_tied_to_the_sources(tmp_path, monkeypatch):
    h = bench.source_hash()
    f = tmp_path / "traffic.txt"
    f.write_text(f"# note: one\nsource_sha256: {h}\ndram_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.stored_traffic() == 12345.0
    f.write_text("source_sha256: 0000\ndram_bytes_per_launch: 12345\n")
    assert bench.stored_traffic() is None


def test_rows_an_early_exit_depends_on():
    # n < K: target and draft rows 0..n; n = K: all 2K + 1 rows
    assert bench.chain_rows_used([0, 8, 3], 8) == 2 + 17 + 8


def test_oracle_rates_reports_both_legs():
    calls = []
    r = bench.oracle_rates(lambda b: calls.append(b), 5, 0.01, 2)
    assert r["single_thread"] > 0 and r["all_cores"] > 0 and r["cores"] == 2
    assert set(calls) <= set(range(5))
