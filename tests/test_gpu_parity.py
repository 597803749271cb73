"""Parity of the CUDA path with the oracle on the same seeded inputs (needs a GPU).

Bars (element by element): page-table slots and Philox words bit-exact; keys/values,
hidden states and logits within max-relative-error 2e-2 (bf16) / 1e-4 (float32),
logits per row; token ids identical wherever the oracle's top-2 margin exceeds 1e-2
and twice the row's measured logit error (see tests/flashmap_harness.py, check_request).
"""

import numpy as np
import pytest
import torch

from oracle import flashmap_ref as ref
from speculative_decoding_block_context_gb300 import _lib as F
from speculative_decoding_block_context_gb300 import synthetic as syn

from .flashmap_harness import TOL, check_request, load_model, max_rel, oracle_batch, oracle_request, run_library, slot_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def built():
    from speculative_decoding_block_context_gb300 import build

    build.build()
    F.lib()


# ---------------------------------------------------------------------- kernels in isolation


def test_philox_words_bit_exact():
    g = torch.Generator().manual_seed(0)
    n = 1 << 20
    seeds = torch.randint(0, 2**63 - 1, (n,), generator=g, dtype=torch.int64)
    ctr = torch.randint(0, 2**32, (n, 4), generator=g, dtype=torch.int64)
    ctr[:4] = torch.tensor([[0, 0, 0, 0], [2**32 - 1] * 4, [1, 2, 3, 4], [5, 6, 7, 8]])
    out = torch.empty((n, 4), dtype=torch.int32, device="cuda")
    normals = torch.empty((n, 4), dtype=torch.float32, device="cuda")
    F.flashmap_debug_philox(seeds.cuda(), ctr.to(torch.int32).cuda(), out, normals)
    torch.cuda.synchronize()
    s = seeds.numpy().astype(np.uint64)
    keys = np.stack([s & np.uint64(0xFFFFFFFF), s >> np.uint64(32)], axis=1)
    want = ref.philox4x32_10(ctr.numpy().astype(np.uint64), keys)
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), want)
    # the Box-Muller normals of the draft noise, within float32 evaluation error
    w = want[:4096].astype(np.uint64)
    n0, n1 = ref.box_muller(w[:, 0], w[:, 1])
    n2, n3 = ref.box_muller(w[:, 2], w[:, 3])
    np.testing.assert_allclose(normals[:4096].cpu().numpy(), np.stack([n0, n1, n2, n3], 1), rtol=2e-5, atol=2e-5)


# Shapes span both ways a tile's k range is split on one SM: thread-block clusters of up
# to 8 CTAs summing through shared memory (at most half as many weight tiles as CTAs,
# e.g. 16 x 4096 -> 4096 in clusters of 8, 16 x 4096 -> 12288 in clusters of 3) and
# stream-K over every CTA with two or three parts per tile summed through the scratch
# (16 x 4096 -> 40960: 320 tiles; 64 x 4096 -> 12288). 200 x 4096 -> 12288 and the last
# four run on SM pairs (tcgen05 cta_group::2, whole 256 x 256 tiles: 48 of them on 48
# pairs, then 5.05, 8.3, 1.26 and 4.1 tiles per pair; ragged rows, and last tiles whose
# second half lies past N); 512 x 1024 -> 4096 and 300 x 512 -> 4800 with 32 and 38
# tiles, the fewest that take the pairs.
@pytest.mark.parametrize("rows,k,n", [(1, 64, 128), (5, 200, 300), (16, 4096, 4096), (37, 384, 1234),
                                      (100, 256, 384), (300, 512, 256), (2048, 1024, 512), (300, 384, 1234),
                                      (513, 4096, 384), (16, 4096, 12288), (16, 12288, 4096), (16, 4096, 40960),
                                      (200, 4096, 12288), (64, 4096, 12288), (2048, 512, 12288), (1000, 256, 40000), (512, 1024, 12288), (300, 384, 40000),
                                      (512, 1024, 4096), (300, 512, 4800)])
def test_linear_bf16_tcgen05(rows, k, n):
    """y = x W^T added onto a nonzero output (the residual stream's mode), against
    float64; a second call on the same inputs gives the same bits (every split tile is
    summed in a fixed order)."""
    g = torch.Generator(device="cuda").manual_seed(rows * 7 + k)
    x = torch.randn((rows, k), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((n, k), generator=g, device="cuda") / k**0.5).to(torch.bfloat16)
    out0 = torch.randn((rows, n), generator=g, device="cuda")
    out = out0.clone()
    F.flashmap_debug_linear(F.BF16, x, w, out)
    out2 = out0.clone()
    F.flashmap_debug_linear(F.BF16, x, w, out2)
    torch.cuda.synchronize()
    want = out0.double().cpu().numpy() + x.double().cpu().numpy() @ w.double().cpu().numpy().T
    assert max_rel(out.cpu().numpy(), want) < 1e-5
    assert torch.equal(out.view(torch.int32), out2.view(torch.int32))


@pytest.mark.parametrize("rows,k,n", [(1, 64, 128), (5, 208, 300), (16, 4096, 4096), (37, 384, 1234),
                                      (100, 256, 384), (300, 512, 256), (2048, 1024, 512), (1024, 512, 12288),
                                      (300, 256, 40000)])
def test_linear_e4m3_tcgen05(rows, k, n):
    """W8A16: w quantized per output channel at call time, expanded to bf16 on chip (the
    last two with 256-row tiles, split over the SMs by stream-K)."""
    g = torch.Generator(device="cuda").manual_seed(rows * 11 + k)
    x = torch.randn((rows, k), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((n, k), generator=g, device="cuda") / k**0.5).to(torch.bfloat16)
    w[min(3, n - 1)] = 0  # an all-zero channel takes scale 1
    out = torch.zeros((rows, n), dtype=torch.float32, device="cuda")
    F.flashmap_debug_linear(F.E4M3, x, w, out)
    torch.cuda.synchronize()
    wq = ref.dequantize(*ref.quantize_e4m3_per_channel(w.float().cpu().numpy()))
    want = x.double().cpu().numpy() @ wq.T
    assert max_rel(out.cpu().numpy(), want) < 1e-5


def test_linear_f32_simt():
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn((7, 300), generator=g, device="cuda")
    w = torch.randn((129, 300), generator=g, device="cuda")
    out = torch.zeros((7, 129), dtype=torch.float32, device="cuda")
    F.flashmap_debug_linear(F.F32, x, w, out)
    torch.cuda.synchronize()
    want = x.double().cpu().numpy() @ w.double().cpu().numpy().T
    assert max_rel(out.cpu().numpy(), want) < 1e-6


# ---------------------------------------------------------------------- whole step


@pytest.fixture(scope="module")
def tiny():
    return load_model("tiny_fp32")


@pytest.fixture(scope="module")
def small():
    return load_model("small_bf16")


def _check_all(st, run, subset, tol):
    report = {}
    outs = oracle_batch(st, run, list(subset))
    for b in subset:
        check_request(st, run, b, outs[b], tol, report)
    return report


def _check_constants(st, tol):
    H = st.cfg["target_hidden"]
    chol = torch.empty((H, H), dtype=torch.float32, device="cuda")
    u = torch.empty(H, dtype=torch.float32, device="cuda")
    hot = torch.empty(st.consts.hot.shape[0], dtype=torch.int64, device="cuda")
    F.flashmap_debug_constants(st.handle, chol, u, hot)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hot.cpu().numpy(), st.consts.hot)
    assert max_rel(u.cpu().numpy(), st.consts.uniform) < tol
    assert max_rel(chol.cpu().numpy(), st.consts.chol) < tol


def test_tiny_fp32_end_to_end(tiny):
    _check_constants(tiny, 1e-5)
    run = run_library("tiny_fp32", tiny)
    assert run.dev_err == 0
    rep = _check_all(tiny, run, range(run.req["bs"]), TOL["f32"])
    assert rep["tokens_checked"] > 0


def test_small_bf16_end_to_end(small):
    _check_constants(small, 1e-2)
    run = run_library("small_bf16", small)
    assert run.dev_err == 0
    _check_all(small, run, range(run.req["bs"]), TOL["bf16"])
    # full-vocabulary logits: the draft logits at their token ids, -inf elsewhere (exact)
    hot = torch.as_tensor(small.consts.hot, device="cuda")
    mask = torch.ones(small.cfg["vocab_size"], dtype=torch.bool, device="cuda")
    mask[hot] = False
    assert torch.isneginf(run.full[:, mask]).all()
    assert torch.equal(run.full[:, hot], run.logits)


@pytest.fixture(scope="module")
def small_kv8():
    return load_model("small_bf16_kv8")


def test_small_e4m3_kv_pool_end_to_end(small_kv8):
    """e4m3 draft KV pool: the written rows are the e4m3 rounding (scale 1) of the
    oracle's keys/values, and the draft with fp8 queries per (request, head) matches
    the oracle run on the stored values."""
    run = run_library("small_bf16_kv8", small_kv8)
    assert run.dev_err == 0
    assert run.pool_t.numel() * 2 == F.flashmap_pool_bytes(dict(small_kv8.cfg, kv_dtype="bf16"), run.req["num_pages"])
    _check_all(small_kv8, run, range(run.req["bs"]), TOL["bf16"])


def test_deferred_window_write_in_the_draft(small):
    """flashmap_draft_block_with_write (flashmap/vllm/model.py, defer_context_kv /
    _prologue): the verify window's committed rows and the anchors through one context
    K/V GEMM. 3 requests x 17 columns take the device-compacted path; slots, out_loc and
    keys/values are checked against the oracle like the separate write's, and the draft
    equals the two-call step's bit for bit."""
    req = syn.make_requests("small_bf16", "cuda")
    run = run_library("small_bf16", small, req=req, deferred=True)
    assert run.dev_err == 0
    _check_all(small, run, range(run.req["bs"]), TOL["bf16"])
    two = run_library("small_bf16", small, req=req)
    assert torch.equal(run.window_loc, two.window_loc)
    assert torch.equal(run.hidden.view(torch.int16), two.hidden.view(torch.int16))
    assert torch.equal(run.tokens, two.tokens)


def test_noise_scale_zero_is_seed_independent(small):
    """noise_scale 0 makes the draft a fixed function of the context: other seeds give
    bitwise the same hidden states, and the oracle agrees."""
    req = syn.make_requests("small_bf16", "cuda")
    a = run_library("small_bf16", small, noise_scale=0.0, req=req)
    req2 = dict(req, seeds=req["seeds"] + 12345)
    b = run_library("small_bf16", small, noise_scale=0.0, req=req2)
    assert torch.equal(a.hidden.view(torch.int16), b.hidden.view(torch.int16))
    o = oracle_request(small, a, 1, noise_scale=0.0)
    K = small.cfg["block_size"]
    assert max_rel(a.hidden[K : 2 * K].float().cpu().numpy(), o["hidden"]) <= TOL["bf16"]


def test_pipeline_wait_timeout_is_reported(small):
    """Every pipeline wait in the kernels is bounded: a wait that runs out sets
    FLASHMAP_DEVERR_TIMEOUT and the kernel returns, leaving the context usable. A probe
    waits 1 ms on an mbarrier that nothing arrives on (no fault, no copy, no MMA); the
    bit comes back through flashmap_get_device_error, which then clears it, and the
    model still drafts."""
    assert F.flashmap_get_device_error(small.handle) == 0
    F.flashmap_debug_wait_timeout(small.handle, 1_000_000)
    torch.cuda.synchronize()
    assert F.flashmap_get_device_error(small.handle) == F.DEVERR["TIMEOUT"]
    assert F.flashmap_get_device_error(small.handle) == 0
    run = run_library("small_bf16", small)
    assert run.dev_err == 0


def test_out_of_range_page_sets_device_error(small):
    """A page id outside the pool is skipped and reported, not dereferenced."""
    req = syn.make_requests("small_bf16", "cuda")
    row = int(req["req_pool_idx"][0])
    req["req_to_page"][row, 0] = req["num_pages"] + 5
    run = run_library("small_bf16", small, req=req)
    assert run.dev_err & F.DEVERR["PAGE"]
    assert int(run.prefill_loc[0][0]) == -1


def test_graph_capture_replays_draft_and_sample(small):
    """The per-step calls allocate nothing and never sync: they capture into a CUDA
    graph whose replay reproduces the eager results."""
    st = small
    cfg = st.cfg
    req = syn.make_requests("small_bf16", "cuda")
    eager = run_library("small_bf16", st, req=req)
    bs, K = req["bs"], cfg["block_size"]
    pool = F.make_pool(eager.pool_t, req["num_pages"], F.BF16)
    ws = torch.empty(F.flashmap_workspace_size(st.handle, bs, 64), dtype=torch.uint8, device="cuda")
    anchor_pos = torch.tensor(req["anchor_pos"], dtype=torch.int32, device="cuda")
    hidden = torch.empty_like(eager.hidden)
    tokens = torch.empty_like(eager.tokens)
    logits = torch.empty_like(eager.logits)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            F.flashmap_draft_block(st.handle, pool, bs, req["anchor_ids"], anchor_pos, req["req_pool_idx"],
                                   req["req_to_page"], req["seeds"], 1.0, hidden, None, ws)
            F.flashmap_sample_block(st.handle, bs, hidden, anchor_pos, req["temperature"], req["greedy"],
                                    req["seeds"], req["step"], tokens, logits, None, ws)
    g.replay()
    torch.cuda.synchronize()
    # the same bits as the eager calls
    assert torch.equal(tokens, eager.tokens)
    assert torch.equal(hidden.view(torch.int16), eager.hidden.view(torch.int16))
    assert torch.equal(logits.view(torch.int32), eager.logits.view(torch.int32))


def _assert_same_bits(a, b, cfg):
    """Two library runs of the same inputs: written pool rows, hidden states, logits,
    the full-vocabulary scatter and tokens bitwise equal."""
    slots = [loc for loc in a.prefill_loc] + [a.anchor_loc]
    if a.window_loc is not None:
        slots.append(a.window_loc[a.window_loc >= 0])
    for i, loc in enumerate(slots):
        s = loc.long()
        for ga, gb in zip(slot_rows(cfg, a.kv, s), slot_rows(cfg, b.kv, s)):
            assert torch.equal(ga.contiguous().view(torch.uint8), gb.contiguous().view(torch.uint8)), f"written rows {i} differ"
    assert torch.equal(a.hidden.view(torch.int16) if a.hidden.dtype == torch.bfloat16 else a.hidden.view(torch.int32),
                       b.hidden.view(torch.int16) if b.hidden.dtype == torch.bfloat16 else b.hidden.view(torch.int32))
    assert torch.equal(a.logits.view(torch.int32), b.logits.view(torch.int32))
    if a.full is not None:
        assert torch.equal(a.full.view(torch.int32), b.full.view(torch.int32))
    assert torch.equal(a.tokens, b.tokens)


def test_load_is_repeatable():
    """Two loads of the same weights derive the same constants bit for bit (the gram
    and the column sums of E are summed in a fixed order) and so draft the same blocks."""
    a = load_model("small_bf16", oracle=False)
    b = load_model("small_bf16", oracle=False)
    H = a.cfg["target_hidden"]
    got = []
    for st in (a, b):
        chol = torch.empty((H, H), dtype=torch.float32, device="cuda")
        u = torch.empty(H, dtype=torch.float32, device="cuda")
        F.flashmap_debug_constants(st.handle, chol, u, None)
        got.append((chol, u))
    torch.cuda.synchronize()
    assert torch.equal(got[0][0].view(torch.int32), got[1][0].view(torch.int32))
    assert torch.equal(got[0][1].view(torch.int32), got[1][1].view(torch.int32))
    req = syn.make_requests("small_bf16", "cuda")
    _assert_same_bits(run_library("small_bf16", a, req=req), run_library("small_bf16", b, req=req), a.cfg)


@pytest.mark.parametrize("workload", ["small_bf16", "tiny_fp32", "small_bf16_3jump", "small_bf16_folded"])
def test_draft_repeats_bit_for_bit(workload):
    """flashmap/vllm/model.py, module docstring: a seeded request drafts the same
    blocks on every run. Two runs of the whole step (context write, draft, sample) on
    the same inputs give the same bits: no result depends on the order in which CTAs
    finish (split GEMM tiles are summed in a fixed order)."""
    st = load_model(workload, oracle=False)
    req = syn.make_requests(workload, "cuda")
    a = run_library(workload, st, req=req)
    b = run_library(workload, st, req=req)
    assert a.dev_err == 0 and b.dev_err == 0
    _assert_same_bits(a, b, st.cfg)


# ---------------------------------------------------------------------- several jumps


@pytest.mark.parametrize("workload,tol", [("tiny_fp32_2jump", 1e-4), ("small_bf16_3jump", 2e-2)])
def test_several_jumps_end_to_end(workload, tol):
    """Drafting in 2 and 3 jumps: the vocabulary-sized state, its posterior and
    linear embeddings, the per-jump modulations and the state update between jumps,
    against the oracle's jump loop (hidden states, logits, tokens where clear)."""
    st = load_model(workload)
    assert st.cfg["num_steps"] > 1
    run = run_library(workload, st)
    assert run.dev_err == 0
    _check_all(st, run, range(run.req["bs"]), tol)


# ---------------------------------------------------------------------- folded-noise eigenbasis


def _check_folded_constants(st, tol):
    """The load-time eigenbasis against the oracle's float64 eigh (reading R9: ascending,
    each eigenvector's largest entry positive): lam / H, x_embed(u) and the projection
    M^T as the GEMM holds it (relative to its largest entry)."""
    H, D = st.cfg["target_hidden"], st.cfg["hidden"]
    Fo = st.consts.extra["folded"]
    var = torch.empty(H, dtype=torch.float32, device="cuda")
    xu = torch.empty(D, dtype=torch.float32, device="cuda")
    proj = torch.empty((D, H), dtype=syn.torch_dtype(st.cfg["act_dtype"]), device="cuda")
    sweeps = F.flashmap_debug_folded(st.handle, var, xu, proj)
    torch.cuda.synchronize()
    assert 0 < sweeps < 60
    np.testing.assert_allclose(var.cpu().numpy(), Fo.variance, rtol=1e-5, atol=1e-7 * Fo.variance.max())
    assert max_rel(xu.cpu().numpy(), Fo.embedded_uniform) < 1e-5
    assert max_rel(proj.float().cpu().numpy(), Fo.proj.T) < tol
    return sweeps


@pytest.mark.parametrize("workload,tol,ctol", [("tiny_fp32_folded", 1e-4, 1e-5), ("small_bf16_folded", 2e-2, 1e-2)])
def test_folded_noise_end_to_end(workload, tol, ctol):
    """noise_path 1: the eigenbasis found at load (float64 one-sided Jacobi) and the
    per-step folded noise (z scaled by gate * rsqrt(sum(lam z^2) / H + eps), one GEMM
    through M onto x_embed(u)) against the oracle's eigh and fold."""
    st = load_model(workload)
    _check_folded_constants(st, ctol)
    run = run_library(workload, st)
    assert run.dev_err == 0
    _check_all(st, run, range(run.req["bs"]), tol)

