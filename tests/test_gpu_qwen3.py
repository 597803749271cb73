"""Parity at the full Qwen3-8B-shaped sizes (target_hidden 4096 x 3 layers, DiT 5 x 4096,
32 x 128 heads, MLP 12288, vocabulary 151936, draft vocabulary 32768), in the launch
configuration the benchmark times. Requests are independent, so the oracle checks a
fixed subset exactly: the shortest and longest contexts and six seeded others."""

import numpy as np
import pytest
import torch

from speculative_decoding_block_context_gb300 import _lib as F

from .flashmap_harness import TOL, check_request, load_model, max_rel, oracle_batch, run_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qwen():
    from speculative_decoding_block_context_gb300 import build

    build.build()
    return load_model("qwen3_8b_bs1")


def subset_of(req, n_random=6, seed=0):
    ctx = np.asarray(req["ctx"])
    picks = {int(np.argmin(ctx)), int(np.argmax(ctx))}
    rng = np.random.default_rng(seed)
    for b in rng.permutation(len(ctx)):
        if len(picks) >= 2 + n_random:
            break
        picks.add(int(b))
    return sorted(picks)


def _run_and_check(qwen, workload, deferred=False):
    from speculative_decoding_block_context_gb300 import synthetic as syn

    req = syn.make_requests(workload, "cuda")
    subset = list(range(req["bs"])) if req["bs"] == 1 else subset_of(req)
    run = run_library(workload, qwen, req=req, check_subset=subset, deferred=deferred)
    assert run.dev_err == 0
    report = {}
    outs = oracle_batch(qwen, run, subset)
    for b in subset:
        check_request(qwen, run, b, outs[b], TOL["bf16"], report)
    print(workload, report)
    # Of the tokens whose oracle margin exceeds 1e-2, the guard against the row's own
    # logit error (margin <= 2 x error) may leave out only a few: measured 0-10% at
    # these sizes (logit errors up to ~0.04 on rows of magnitude ~10); 15% (+1) bounds it.
    assert report["tokens_guarded"] <= 0.15 * report["tokens_margin_ok"] + 1, report
    return run, report


def test_qwen3_bs1_repeats_bit_for_bit(qwen):
    """The batch-1 step (2048-position prefill, verify-window write, draft, sample) run
    twice on the same inputs gives the same bits (flashmap/vllm/model.py, module
    docstring: a seeded request drafts the same blocks on every run)."""
    from speculative_decoding_block_context_gb300 import synthetic as syn

    from .test_gpu_parity import _assert_same_bits

    req = syn.make_requests("qwen3_8b_bs1", "cuda")
    a = run_library("qwen3_8b_bs1", qwen, req=req)
    b = run_library("qwen3_8b_bs1", qwen, req=req)
    assert a.dev_err == 0 and b.dev_err == 0
    _assert_same_bits(a, b, qwen.cfg)


def test_qwen3_constants(qwen):
    H = qwen.cfg["target_hidden"]
    chol = torch.empty((H, H), dtype=torch.float32, device="cuda")
    u = torch.empty(H, dtype=torch.float32, device="cuda")
    hot = torch.empty(qwen.consts.hot.shape[0], dtype=torch.int64, device="cuda")
    F.flashmap_debug_constants(qwen.handle, chol, u, hot)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hot.cpu().numpy(), qwen.consts.hot)
    assert max_rel(u.cpu().numpy(), qwen.consts.uniform) < 1e-4
    assert max_rel(chol.cpu().numpy(), qwen.consts.chol) < 1e-2  # L is stored in bf16


def test_qwen3_bs1_prefill_window_draft_sample(qwen):
    _run_and_check(qwen, "qwen3_8b_bs1")


def test_qwen3_bs1_deferred_window_write(qwen):
    """The verify-window write deferred into the draft (one context K/V GEMM over the
    17 window rows and the anchor; the window is below the compaction threshold)."""
    _run_and_check(qwen, "qwen3_8b_bs1", deferred=True)


def test_qwen3_bs32_ragged_contexts(qwen):
    _run_and_check(qwen, "qwen3_8b_bs32")


def test_qwen3_e4m3_kv_pool_bs32(qwen):
    """The batch-32 workload over an e4m3 draft KV pool: the same weights loaded with
    kv_dtype e4m3 (the oracle reads the pool's e4m3 values and quantizes its queries
    per (request, head) as the fp8 cross-attention does)."""
    import dataclasses

    from speculative_decoding_block_context_gb300 import synthetic as syn

    cfg8 = syn.model_config("qwen3_8b_bs32_kv8")
    st8 = dataclasses.replace(qwen, cfg=cfg8, handle=F.flashmap_load_weights(cfg8, qwen.W, qwen.E, qwen.LM, qwen.rank))
    run, _ = _run_and_check(st8, "qwen3_8b_bs32_kv8")
    del run, st8
    torch.cuda.empty_cache()


def test_qwen3_e4m3_kv_pool_bs128(qwen):
    """The batch-128 workload (log-uniform contexts 16..32768, verify-window write,
    full-vocabulary scatter) over an e4m3 pool: the window rows are written through the
    e4m3 store (values channel-major per (page, head) block), then read back by the
    oracle and by the e4m3 cross-attention."""
    import dataclasses

    from speculative_decoding_block_context_gb300 import synthetic as syn

    cfg8 = syn.model_config("qwen3_8b_bs128_kv8")
    st8 = dataclasses.replace(qwen, cfg=cfg8, handle=F.flashmap_load_weights(cfg8, qwen.W, qwen.E, qwen.LM, qwen.rank))
    run, _ = _run_and_check(st8, "qwen3_8b_bs128_kv8")
    del run, st8
    torch.cuda.empty_cache()


def test_qwen3_two_jumps_bs1(qwen):
    """Drafting in two jumps on the printed grid (0, 0.8172569274902344, 1) at the full
    sizes: the state is 151936
    wide per row, read through E (4096) as posterior and state, and moved by the
    full-vocabulary head between the jumps. Same weights, loaded with num_steps 2."""
    import dataclasses

    from speculative_decoding_block_context_gb300 import synthetic as syn

    cfg2 = syn.model_config("qwen3_8b_bs1_2jump")
    assert cfg2["num_steps"] == 2
    st2 = dataclasses.replace(qwen, cfg=cfg2, handle=F.flashmap_load_weights(cfg2, qwen.W, qwen.E, qwen.LM, qwen.rank))
    run, _ = _run_and_check(st2, "qwen3_8b_bs1_2jump")
    del run, st2
    torch.cuda.empty_cache()


def test_qwen3_folded_noise_bs1(qwen):
    """The folded-noise eigenbasis at the full sizes: the 4096 x 4096 gram's float64
    Jacobi eigenpairs at load against the oracle's eigh (lam / H, x_embed(u), the
    projection), then the batch-1 draft through the folded GEMM. Same weights, loaded
    with noise_path 1; the oracle adds its fold to the constants it already has."""
    import dataclasses
    import time

    from oracle import flashmap_ref as ref
    from speculative_decoding_block_context_gb300 import synthetic as syn

    from .test_gpu_parity import _check_folded_constants

    cfgf = syn.model_config("qwen3_8b_bs1_folded")
    t0 = time.perf_counter()
    handle = F.flashmap_load_weights(cfgf, qwen.W, qwen.E, qwen.LM, qwen.rank)
    torch.cuda.synchronize()
    load_s = time.perf_counter() - t0
    consts = dataclasses.replace(qwen.consts, extra=dict(qwen.consts.extra))
    consts.extra["folded"] = ref.folded_noise(ref.Config.from_dict(cfgf), qwen.Wnp, consts)
    stf = dataclasses.replace(qwen, cfg=cfgf, handle=handle, consts=consts)
    sweeps = _check_folded_constants(stf, 1e-2)
    print("folded load", round(load_s, 2), "s,", sweeps, "Jacobi sweeps")
    run, _ = _run_and_check(stf, "qwen3_8b_bs1_folded")
    del run, stf
    torch.cuda.empty_cache()


def test_qwen3_fp8_weights_bs64_greedy(qwen):
    """Config 5: e4m3 DiT weights with per-channel scales, bf16 activations; the oracle
    runs on the dequantized weights. The bf16 model of the other tests stays loaded."""
    fp8 = load_model("qwen3_8b_fp8_bs64")
    run, _ = _run_and_check(fp8, "qwen3_8b_fp8_bs64")
    del run, fp8  # the handle frees the model's arena
    torch.cuda.empty_cache()


@pytest.mark.parametrize("deferred", [False, True], ids=["two_calls", "deferred_write"])
def test_qwen3_bs128_window_and_full_vocab_scatter(qwen, deferred):
    """Batch 128 with a 17-column verify window (1..16 committed): the separate write
    call, or the write deferred into the draft (2176 window rows, compacted on the
    device, and the 128 anchors through one context K/V GEMM)."""
    run, _ = _run_and_check(qwen, "qwen3_8b_bs128", deferred=deferred)
    hot = torch.as_tensor(qwen.consts.hot, device="cuda")
    mask = torch.ones(qwen.cfg["vocab_size"], dtype=torch.bool, device="cuda")
    mask[hot] = False
    for r0 in range(0, run.full.shape[0], 256):
        blk = run.full[r0 : r0 + 256]
        assert torch.isneginf(blk[:, mask]).all()
        assert torch.equal(blk[:, hot], run.logits[r0 : r0 + 256])


@pytest.mark.parametrize("workload,subset", [("qwen3_8b_bs1_tree4", [0]), ("qwen3_8b_bs32_tree4", None)])
def test_qwen3_tree_drafting(qwen, workload, subset):
    """Tree drafting at the full sizes, as the benchmark runs it: 4 candidate blocks per
    request from candidate-keyed noise, greedy tokens, the verify tree of width 16.
    Candidates of the checked requests (batch 32: the shortest and longest contexts
    and one other) against the oracle; every checked request's tree against the
    oracle's trie over those tokens."""
    from speculative_decoding_block_context_gb300 import synthetic as syn

    from .flashmap_harness import check_candidates, run_candidates

    req = syn.make_requests(workload, "cuda")
    sub = subset if subset is not None else subset_of(req, n_random=1)
    run = run_library(workload, qwen, req=req, check_subset=sub)
    assert run.dev_err == 0
    n, width = req["tree"]
    out = run_candidates(qwen, run, n, width)
    counts = check_candidates(qwen, run, n, width, TOL["bf16"], 1e-2, sub, out)
    print(workload, counts)
    assert counts["trees"] == len(sub)
