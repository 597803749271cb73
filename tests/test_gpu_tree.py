"""The verify tree kernel against the oracle's trie, bit-exact, on seeded candidate
blocks: small alphabets (many shared prefixes and repeated candidates), all-distinct
candidates, cuts below and above the trie's size (padding), and the limits."""

import numpy as np
import pytest
import torch

from oracle import flashmap_ref as ref
from speculative_decoding_block_context_gb300 import _lib as F

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_block_context_gb300 import build

    build.build()
    F.lib()


@pytest.mark.parametrize("bs,n,k,width,alphabet,seed", [
    (4, 8, 16, 64, 2, 0),      # binary tokens: deep shared prefixes
    (3, 16, 16, 32, 3, 1),
    (2, 64, 16, 128, 4, 2),    # the most candidates, 1024 nodes
    (5, 4, 6, 100, 5, 3),      # fewer nodes than width - 1: padding
    (2, 1, 16, 8, 151936, 4),  # one candidate: a chain
    (3, 32, 8, 17, 151936, 5), # all distinct at depth 0
    (1, 64, 16, 1025, 2, 6),   # the widest tree
])
def test_tree_matches_oracle(bs, n, k, width, alphabet, seed):
    g = torch.Generator().manual_seed(seed)
    cand = torch.randint(0, alphabet, (bs, n, k), generator=g, dtype=torch.int64)
    if n > 2:
        cand[:, 1] = cand[:, 0]  # a repeated candidate
    m = width - 1
    tokens = torch.full((bs, m), -7, dtype=torch.int64, device="cuda")
    ids = torch.full((bs, m), -7, dtype=torch.int64, device="cuda")
    stats = torch.full((bs, 2), -7, dtype=torch.int64, device="cuda")
    F.flashmap_build_tree(cand.cuda(), width, tokens, ids, stats)
    torch.cuda.synchronize()
    for b in range(bs):
        wt, wi, ws = ref.build_tree(cand[b].numpy(), width)
        np.testing.assert_array_equal(tokens[b].cpu().numpy(), wt)
        np.testing.assert_array_equal(ids[b].cpu().numpy(), wi)
        np.testing.assert_array_equal(stats[b].cpu().numpy(), ws)


def test_tree_refuses_out_of_range_shapes():
    cand = torch.zeros((1, 65, 2), dtype=torch.int64, device="cuda")
    out = torch.zeros((1, 8), dtype=torch.int64, device="cuda")
    st = torch.zeros((1, 2), dtype=torch.int64, device="cuda")
    with pytest.raises(F.FlashmapError):
        F.flashmap_build_tree(cand, 9, out, out, st)  # 65 candidates
    cand = torch.zeros((1, 4, 2), dtype=torch.int64, device="cuda")
    with pytest.raises(F.FlashmapError):
        F.flashmap_build_tree(cand, 1, out, out, st)  # width 1


# ------------------------------------------------------------------ tree drafting


@pytest.mark.parametrize("workload,n,width,tol,margin", [
    ("small_bf16", 3, 12, 2e-2, 1e-2),
    ("tiny_fp32", 8, 16, 1e-4, 1e-4),
    ("small_bf16_folded", 3, 12, 2e-2, 1e-2),  # candidates on the folded-noise path
    # 2, 4 and 8 candidates: a CTA's warps serve 2 or 4 candidate blocks from one read
    # of each K/V block (8: two groups of 4)
    ("small_bf16", 2, 8, 2e-2, 1e-2),
    ("small_bf16", 4, 16, 2e-2, 1e-2),
    ("small_bf16", 8, 24, 2e-2, 1e-2),
    ("small_bf16_kv8", 4, 16, 2e-2, 1e-2),  # e4m3 pool
    ("small_bf16_kv8", 2, 8, 2e-2, 1e-2),
])
def test_candidate_draft_and_tree_against_the_oracle(workload, n, width, tol, margin):
    """Candidate blocks per request: every block's hidden states and logits match the
    oracle's draft with candidate-keyed noise (candidate 0 being the single draft),
    greedy tokens match wherever the oracle's top-2 margin is clear, and every
    request's tree is the oracle's trie over those tokens (see check_candidates)."""
    from .flashmap_harness import check_candidates, load_model, max_rel, run_candidates, run_library

    st = load_model(workload)
    run = run_library(workload, st)  # the pool now holds every written row
    out = run_candidates(st, run, n, width)
    bs, K = run.req["bs"], st.cfg["block_size"]
    # candidate 0 is the single draft (up to rounding: the candidate draft's GEMMs run on
    # n times the rows, so their tiles are split differently)
    h0 = out[0].view(bs, n, K, -1)[:, 0].reshape(bs * K, -1).float().cpu().numpy()
    assert max_rel(h0, run.hidden.float().cpu().numpy()) < (1e-2 if tol > 1e-3 else 1e-5)
    counts = check_candidates(st, run, n, width, tol, margin, range(bs), out)
    print(workload, n, counts)
    assert counts["trees"] == bs
