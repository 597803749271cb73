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


@pytest.mark.parametrize("workload,n,width,tol,margin,min_trees", [
    ("small_bf16", 3, 12, 2e-2, 1e-2, 0),  # bf16: tokens compared where the margin is clear
    ("tiny_fp32", 8, 16, 1e-4, 1e-4, 1),   # fp32: whole trees compared
    ("small_bf16_folded", 3, 12, 2e-2, 1e-2, 0),  # candidates on the folded-noise path
    # 2, 4 and 8 candidates: a CTA's warps serve 2 or 4 candidate blocks from one read
    # of each K/V block (8: two groups of 4)
    ("small_bf16", 2, 8, 2e-2, 1e-2, 0),
    ("small_bf16", 4, 16, 2e-2, 1e-2, 0),
    ("small_bf16", 8, 24, 2e-2, 1e-2, 0),
    ("small_bf16_kv8", 4, 16, 2e-2, 1e-2, 0),  # e4m3 pool
    ("small_bf16_kv8", 2, 8, 2e-2, 1e-2, 0),
])
def test_candidate_draft_and_tree_against_the_oracle(workload, n, width, tol, margin, min_trees):
    margin_min = margin
    """Candidate blocks per request: every block's hidden states and logits match the
    oracle's draft with candidate-keyed noise (candidate 0 being the single draft),
    their greedy tokens match wherever the oracle's top-2 margin is clear, and each
    request whose candidates are all clear gets the oracle's tree, bit-exact."""
    from oracle import flashmap_ref as ref
    from speculative_decoding_block_context_gb300 import synthetic as syn

    from .flashmap_harness import load_model, max_rel, oracle_contexts, run_library

    st = load_model(workload)
    run = run_library(workload, st)  # the pool now holds every written row
    req, cfg = run.req, st.cfg
    bs, K, D = req["bs"], cfg["block_size"], cfg["hidden"]
    dt = syn.torch_dtype(cfg["act_dtype"])
    pool = F.make_pool(run.pool_t, req["num_pages"], F.DTYPE_CODES[cfg["kv_dtype"]])
    ws = torch.empty(F.flashmap_workspace_size(st.handle, bs * n, bs * (K + 1)), dtype=torch.uint8, device="cuda")
    hidden = torch.empty((bs * n * K, D), dtype=dt, device="cuda")
    anchor_pos = torch.tensor(req["anchor_pos"], dtype=torch.int32, device="cuda")
    F.flashmap_draft_candidates(st.handle, pool, bs, n, req["anchor_ids"], anchor_pos, req["req_pool_idx"],
                                req["req_to_page"], req["seeds"], 1.0, hidden, None, ws)
    # greedy tokens of every block: the sampler over bs * n blocks
    rep = lambda t: t.repeat_interleave(n)
    vd = st.consts.hot.shape[0]
    tokens = torch.empty(bs * n * K, dtype=torch.int64, device="cuda")
    logits = torch.empty((bs * n * K, vd), dtype=torch.float32, device="cuda")
    F.flashmap_sample_block(st.handle, bs * n, hidden, rep(anchor_pos), torch.zeros(bs * n, device="cuda"),
                            torch.ones(bs * n, dtype=torch.uint8, device="cuda"), rep(req["seeds"]), 0, tokens,
                            logits, None, ws)
    t_out = torch.empty((bs, width - 1), dtype=torch.int64, device="cuda")
    i_out = torch.empty((bs, width - 1), dtype=torch.int64, device="cuda")
    s_out = torch.empty((bs, 2), dtype=torch.int64, device="cuda")
    F.flashmap_build_tree(tokens.view(bs, n, K), width, t_out, i_out, s_out)
    torch.cuda.synchronize()
    assert F.flashmap_get_device_error(st.handle) == 0
    # candidate 0 is the single draft (up to the GEMMs' atomic summation order)
    h = hidden.float().view(bs, n, K, D).cpu().numpy()
    assert max_rel(h[:, 0].reshape(bs * K, D), run.hidden.float().cpu().numpy()) < max(tol, 1e-2 if tol > 1e-3 else 1e-5)
    _, ctxs, ps, seeds = oracle_contexts(st, run, list(range(bs)))
    ocfg = st.oracle_cfg()
    blocks = [(i, c) for i in range(bs) for c in range(n)]
    want = ref.draft_requests(ocfg, st.Wnp, st.consts, [ctxs[i] for i, _ in blocks], [ps[i] for i, _ in blocks],
                              [seeds[i] for i, _ in blocks], 1.0, [c for _, c in blocks])
    trees_checked = 0
    for b in range(bs):
        otok = []
        clear = True
        for c in range(n):
            assert max_rel(h[b, c], want[b * n + c]) <= tol
            lg = ref.head_logits(st.consts, want[b * n + c])
            got_lg = logits.view(bs, n, K, vd)[b, c].cpu().numpy()
            assert max(max_rel(got_lg[r], lg[r]) for r in range(K)) <= tol
            tok, _, margin = ref.sample_rows(lg, [0.0] * K, [1] * K, [seeds[b]] * K, ps[b] + 1 + np.arange(K), 0,
                                             st.consts.hot)
            got = tokens.view(bs, n, K)[b, c].cpu().numpy()
            sure = margin > margin_min
            np.testing.assert_array_equal(got[sure], tok[sure])
            clear &= bool(sure.all())
            otok.append(tok)
        if clear:  # the oracle's own candidates give the same tree
            wt, wi, wst = ref.build_tree(np.stack(otok), width)
            np.testing.assert_array_equal(t_out[b].cpu().numpy(), wt)
            np.testing.assert_array_equal(i_out[b].cpu().numpy(), wi)
            np.testing.assert_array_equal(s_out[b].cpu().numpy(), wst)
            trees_checked += 1
    print(workload, "trees checked against the oracle:", trees_checked, "of", bs)
    assert trees_checked >= min_trees
