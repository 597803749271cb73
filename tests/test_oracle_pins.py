"""Pins of the oracle to things other than itself: published vectors and printed
constants, closed forms, library routines, brute force and statistical laws.

Each test names what fixes the function; none re-types the oracle's formula."""

import math
import os

import numpy as np
import pytest
import scipy.stats as st

from oracle import flashmap_ref as ref
from speculative_decoding_block_context_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# --------------------------------------------------------------------- Philox


def test_philox_known_answer_vectors():
    """Random123's published Philox4x32-10 known-answer vectors."""
    rows = _rows("philox_kat.txt")
    ctr = np.array([[int(x, 16) for x in r[0:4]] for r in rows], dtype=np.uint64)
    key = np.array([[int(x, 16) for x in r[4:6]] for r in rows], dtype=np.uint64)
    want = np.array([[int(x, 16) for x in r[6:10]] for r in rows], dtype=np.uint32)
    np.testing.assert_array_equal(ref.philox4x32_10(ctr, key), want)


def test_uniform_map_exact_in_float32_and_open_interval():
    w = np.array([0, 1, 511, 512, 0x7FFFFFFF, 0xFFFFFFFF], dtype=np.uint64)
    u = ref.word_to_uniform(w)
    assert u[0] == 2.0**-24 and u[-1] == 1.0 - 2.0**-24
    assert np.all((u > 0) & (u < 1))
    np.testing.assert_array_equal(u.astype(np.float32).astype(np.float64), u)


def test_draft_normals_law():
    """Box-Muller output is N(0, 1): KS test, moments, no column correlation."""
    z = ref.draft_normals(12345, np.arange(4000), 64)
    x = z.reshape(-1)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1) < 0.01
    assert st.kstest(x, "norm").pvalue > 1e-3
    c = np.corrcoef(z[:, :8].T)
    assert np.max(np.abs(c - np.eye(8))) < 0.06


def test_draft_normals_keying():
    """Rows depend only on (seed, position): the same slot position under the same
    seed gives the same noise, another seed or position does not."""
    a = ref.draft_normals(7, [10, 11, 12], 16)
    b = ref.draft_normals(7, [12, 10], 16)
    np.testing.assert_array_equal(a[2], b[0])
    np.testing.assert_array_equal(a[0], b[1])
    assert not np.allclose(ref.draft_normals(8, [10], 16), a[:1])


def test_gumbel_law():
    g = np.concatenate([ref.gumbel_noise(3, p, 5, 64) for p in range(1500)])
    assert st.kstest(g, "gumbel_r").pvalue > 1e-3


# --------------------------------------------------------------------- constants


def test_jump_grids_printed_constants():
    for r in _rows("jump_grids.txt"):
        grid = [float(x) for x in r[1:]]
        assert ref.DEFAULT_JUMP_GRIDS[r[0]] == grid
        assert grid[0] == 0.0 and grid[-1] == 1.0
        assert all(a < b for a, b in zip(grid, grid[1:]))


def test_context_row_bytes_printed_value():
    """The pages' 48 KB per committed row: every layer's key and value, D wide."""
    for L, D, el, want in (map(int, r) for r in _rows("context_row_bytes.txt")):
        k, v = np.zeros((L, 1, 1, D)), np.zeros((L, 1, 1, D))  # (L, n, heads, hd)
        assert (k.size + v.size) * el == want


# --------------------------------------------------------------------- RoPE


def test_rope_closed_form_rotation_and_pairing():
    hd, theta = 16, 1e4
    for pos in (0, 1, 7, 1000):
        ang = ref.rope_angles([pos], hd, theta)[0].astype(np.float64)
        for i in range(hd // 2):
            x = np.zeros((1, 1, hd))
            x[0, 0, 2 * i] = 1.0
            y = ref.apply_rope(x, [pos], theta)[0, 0]
            want = np.zeros(hd)
            want[2 * i], want[2 * i + 1] = math.cos(ang[i]), math.sin(ang[i])
            np.testing.assert_allclose(y, want, atol=1e-15)
    # the angle of pair i is p * theta^(-2i/hd) up to float32 rounding
    ang = ref.rope_angles([3], 8, 10000.0)[0]
    np.testing.assert_allclose(ang, [3 * 10000 ** (-2 * i / 8) for i in range(4)], rtol=1e-6)


def test_rope_norm_and_relative_position():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 2, 32))
    k = rng.standard_normal((1, 2, 32))
    qr = ref.apply_rope(q, [5], 1e4)
    np.testing.assert_allclose(np.linalg.norm(qr, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-13)
    # <R_p q, R_p' k> depends on p - p' only (small positions: float32 angles exact enough)
    d1 = np.sum(ref.apply_rope(q, [9], 1e4) * ref.apply_rope(k, [4], 1e4), axis=-1)
    d2 = np.sum(ref.apply_rope(q, [25], 1e4) * ref.apply_rope(k, [20], 1e4), axis=-1)
    np.testing.assert_allclose(d1, d2, rtol=1e-5)


# --------------------------------------------------------------------- norms etc.


def test_rms_norm_closed_forms():
    w = np.array([1.0, 2.0, 3.0, 4.0])
    x = np.full(4, -3.0)  # rms 3: scale 1/3 per unit weight (eps -> 0)
    np.testing.assert_allclose(ref.rms_norm(x, w, 0.0), -w, rtol=1e-15)
    rng = np.random.default_rng(1)
    y = rng.standard_normal(64)
    # unit weights, eps 0: norm of the output is sqrt(n)
    assert abs(np.linalg.norm(ref.rms_norm(y, np.ones(64), 0.0)) - 8.0) < 1e-12
    # scale invariance (eps 0) and the eps limit at zero input
    np.testing.assert_allclose(ref.rms_norm(5 * y, 1, 0.0), ref.rms_norm(y, 1, 0.0), rtol=1e-13)
    assert np.all(ref.rms_norm(np.zeros(8), 1.0, 1e-6) == 0)


def test_layer_norm_against_zscore():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 50)) * 4 + 1
    np.testing.assert_allclose(ref.layer_norm(x, 0.0), st.zscore(x, axis=-1), rtol=1e-12)


def test_gelu_silu_library_forms():
    x = np.linspace(-6, 6, 101)
    np.testing.assert_allclose(ref.gelu(x), x * st.norm.cdf(x), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(ref.silu(x), x * (1 / (1 + np.exp(-x))), rtol=1e-15)


def test_time_embedding_at_zero_and_one():
    """t = 0: features cos(0) = 1 (first half), sin(0) = 0 (second half); with identity
    linears and zero biases the output is SiLU of those features."""
    Te = C = 8
    I, z = np.eye(8), np.zeros(8)
    out = ref.time_embedding(0.0, I, z, I, z, Te, 1000.0)
    np.testing.assert_allclose(out, ref.silu(np.array([1.0] * 4 + [0.0] * 4)), rtol=1e-15)
    out1 = ref.time_embedding(1.0, I, z, I, z, Te, 1000.0)
    half = 4
    a = 1000.0 * np.array([10000 ** (-i / half) for i in range(half)])
    np.testing.assert_allclose(out1, ref.silu(np.concatenate([np.cos(a), np.sin(a)])), rtol=1e-12)


# --------------------------------------------------------------------- attention


def _attention_brute(q, k, v):
    nq, nh, hd = q.shape
    out = np.zeros_like(q)
    for h in range(nh):
        for i in range(nq):
            s = [sum(q[i, h, d] * k[j, h, d] for d in range(hd)) / math.sqrt(hd) for j in range(k.shape[0])]
            e = [math.exp(x) for x in s]
            tot = sum(e)
            for d in range(hd):
                out[i, h, d] = sum(e[j] * v[j, h, d] for j in range(k.shape[0])) / tot
    return out


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((3, 2, 4)), rng.standard_normal((5, 2, 4)), rng.standard_normal((5, 2, 4))
    np.testing.assert_allclose(ref.attention(q, k, v), _attention_brute(q, k, v), rtol=1e-12)


def test_attention_degenerate_contexts():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((4, 2, 8))
    k1, v1 = rng.standard_normal((1, 2, 8)), rng.standard_normal((1, 2, 8))
    # one position: the output is that position's value whatever the query
    np.testing.assert_allclose(ref.attention(q, k1, v1), np.broadcast_to(v1, (4, 2, 8)), rtol=1e-14)
    # identical keys: the output is the mean value
    k = np.broadcast_to(k1, (6, 2, 8))
    v = rng.standard_normal((6, 2, 8))
    np.testing.assert_allclose(ref.attention(q, k, v), np.broadcast_to(v.mean(0), (4, 2, 8)), rtol=1e-12)


# --------------------------------------------------------------------- model-level


def _tiny(**over):
    from speculative_decoding_block_context_gb300 import synthetic as syn

    d = syn.model_config("tiny_fp32")
    d.update(over)
    cfg = ref.Config.from_dict(d)
    W, E, LM, rank = syn.make_model(d, "cpu")
    W = {k: v.float().numpy() for k, v in W.items()}
    return cfg, W, E.float().numpy(), LM.float().numpy(), rank.numpy()


@pytest.fixture(scope="module")
def tiny():
    cfg, W, E, LM, rank = _tiny()
    return cfg, W, E, LM, rank, ref.load_constants(cfg, W, E, LM, rank)


def test_cholesky_identity(tiny):
    cfg, W, E, LM, rank, C = tiny
    G = E.astype(np.float64).T @ E.astype(np.float64)
    assert np.linalg.norm(C.chol @ C.chol.T - G) / np.linalg.norm(G) < 1e-12
    assert np.allclose(C.chol, np.tril(C.chol)) and np.all(np.diag(C.chol) > 0)


def test_noise_law_matches_embedding_covariance():
    """z L^T ~ N(0, E^T E) (modeling_flashmap.py, target_constants). A gram far from a
    multiple of the identity makes a transposed factor (L^T L) fail."""
    rng = np.random.default_rng(5)
    V, H, N = 512, 24, 60000
    E = rng.standard_normal((V, H)) @ (rng.standard_normal((H, H)) + 2 * np.eye(H)) * 0.05
    L = np.linalg.cholesky(E.T @ E)
    z = ref.draft_normals(99, np.arange(N), H)
    y = z @ L.T
    S = y.T @ y / N
    G = E.T @ E
    assert np.linalg.norm(S - G) / np.linalg.norm(G) < 0.05
    assert np.linalg.norm(L.T @ L - G) / np.linalg.norm(G) > 0.2  # the test can tell
    # the direct draw x0 @ E, x0 ~ N(0, I_V), has the same covariance
    x0 = rng.standard_normal((N, V))
    Y = x0 @ E
    S2 = Y.T @ Y / N
    assert np.linalg.norm(S - S2) / np.linalg.norm(G) < 0.07


def test_fold_identity(tiny):
    """flashmap/sglang/model.py, _fold_lm_head: no nonlinearity between the DiT head
    and the LM head, so LM[hot] (W_head h + b_head) == W_f h + b_f."""
    cfg, W, E, LM, rank, C = tiny
    h = np.random.default_rng(6).standard_normal((3, cfg.hidden))
    two_step = (h @ W["head.weight"].astype(np.float64).T + W["head.bias"]) @ LM[C.hot].astype(np.float64).T
    np.testing.assert_allclose(ref.head_logits(C, h), two_step, rtol=1e-10, atol=1e-12)


def test_uniform_constant_is_embedded_uniform_posterior(tiny):
    """modeling_flashmap.py, target_constants: the uniform posterior (1/V each) times E,
    through state_norm."""
    cfg, W, E, LM, rank, C = tiny
    post = np.full(cfg.vocab_size, 1.0 / cfg.vocab_size) @ E.astype(np.float64)
    rms = np.sqrt(np.mean(post**2) + cfg.rms_norm_eps)
    np.testing.assert_allclose(C.uniform, post / rms * W["state_norm.weight"], rtol=1e-12)


def test_draft_vocabulary(tiny):
    cfg, W, E, LM, rank, C = tiny
    assert len(C.hot) == cfg.draft_vocab_size and np.all(np.diff(C.hot) > 0)
    assert set(C.hot) == set(rank[: cfg.draft_vocab_size])
    full = ref.draft_vocabulary(ref.Config.from_dict({**cfg.__dict__, "draft_vocab_size": 0}), rank)
    np.testing.assert_array_equal(full, np.arange(cfg.vocab_size))


def test_modulations_zero_adaln_gives_identity_modulation():
    cfg, W, E, LM, rank = _tiny()
    for k in W:
        if "adaln.linear" in k:
            W[k] = np.zeros_like(W[k])
    mods, final, _ = ref.jump_conditioning(cfg, W, 0.0, 1.0)
    assert np.all(mods[:, 0::3] == 1) and np.all(mods[:, 1::3] == 0) and np.all(mods[:, 2::3] == 0)
    assert np.all(final[0] == 1) and np.all(final[1] == 0)


def test_draft_zero_gates_reduces_to_embedding():
    """With every AdaLN zeroed, each gated residual vanishes: the draft output is the
    plain LayerNorm of the noise embedding (a dropped gate or residual fails)."""
    cfg, W, E, LM, rank = _tiny()
    for k in W:
        if "adaln.linear" in k:
            W[k] = np.zeros_like(W[k])
    C = ref.load_constants(cfg, W, E, LM, rank)
    p = 10
    rng = np.random.default_rng(7)
    kc = rng.standard_normal((cfg.num_layers, p + 1, cfg.num_heads, cfg.head_dim))
    out = ref.draft_request(cfg, W, C, kc, kc, p, seed=42)
    pos = p + 1 + np.arange(cfg.block_size)
    x0 = ref.noise_embedding(cfg, W, C, 42, pos, 1.0)
    np.testing.assert_allclose(out, ref.layer_norm(x0, cfg.layer_norm_eps), rtol=1e-12)


def test_draft_noise_scale_zero_is_seed_independent(tiny):
    cfg, W, E, LM, rank, C = tiny
    p = 5
    rng = np.random.default_rng(8)
    kc = rng.standard_normal((cfg.num_layers, p + 1, cfg.num_heads, cfg.head_dim))
    a = ref.draft_request(cfg, W, C, kc, kc, p, seed=1, noise_scale=0.0)
    b = ref.draft_request(cfg, W, C, kc, kc, p, seed=2, noise_scale=0.0)
    np.testing.assert_array_equal(a, b)
    c = ref.draft_request(cfg, W, C, kc, kc, p, seed=1)
    assert not np.allclose(a, c)


# --------------------------------------------------------------------- slots


def test_write_locations_brute_force_page_walk():
    rng = np.random.default_rng(9)
    P, rows, pages = 4, 5, 40
    r2p = rng.permutation(pages)[: rows * 8].reshape(rows, 8)
    start = np.array([0, 3, 13, 7])
    commit = np.array([5, 0, 2, 5])
    idx = np.array([2, 0, 4, 1])
    out = ref.write_locations(start, commit, 5, idx, r2p, P)
    for b in range(4):
        # walk the request's pages one slot at a time
        walk = [int(r2p[idx[b], q]) * P + o for q in range(8) for o in range(P)]
        for c in range(5):
            want = walk[start[b] + c] if c < commit[b] else -1
            assert out[b, c] == want


# --------------------------------------------------------------------- sampling


def test_sampling_greedy_and_ties():
    lg = np.array([[0.1, 0.5, 0.5, -1.0], [3.0, 3.0, 3.0, 3.0]])
    hot = np.array([10, 20, 30, 40])
    tok, idx, _ = ref.sample_rows(lg, [0, -1], [1, 0], [1, 2], [5, 6], 0, hot)
    assert list(idx) == [1, 0] and list(tok) == [20, 10]


def test_gumbel_max_law_chi_square():
    """Gumbel-max draws are distributed as softmax(l / T)."""
    l = np.array([0.3, -1.0, 1.2, 0.0, 0.7, -0.4])
    T, n = 0.7, 20000
    counts = np.zeros(len(l))
    rows = np.tile(l, (n, 1))
    seeds = np.arange(n) * 7919 + 3
    _, idx, _ = ref.sample_rows(rows, [T] * n, [0] * n, seeds, np.arange(n) % 97, 11, np.arange(6))
    for j in idx:
        counts[j] += 1
    p = np.exp(l / T) / np.exp(l / T).sum()
    assert st.chisquare(counts, n * p).pvalue > 1e-3


def test_sampling_row_independence():
    rng = np.random.default_rng(10)
    lg = rng.standard_normal((5, 50))
    args = dict(temperature=[1.0] * 5, greedy=[0, 1, 0, 0, 1], seeds=[1, 2, 3, 4, 5],
                positions=[9, 9, 10, 11, 12], step=4, hot=np.arange(50))
    t1, _, _ = ref.sample_rows(lg, **args)
    lg2 = lg.copy()
    lg2[[0, 1, 3]] = rng.standard_normal((3, 50))
    args2 = dict(args, seeds=[9, 2, 3, 8, 5])
    t2, _, _ = ref.sample_rows(lg2, **args2)
    assert t1[2] == t2[2] and t1[4] == t2[4]


def test_full_logits_minus_inf_outside_draft_vocab():
    lg = np.array([[1.0, 2.0, 3.0]])
    full = ref.full_logits(lg, np.array([1, 4, 6]), 8)
    assert np.all(np.isneginf(full[0, [0, 2, 3, 5, 7]]))
    np.testing.assert_array_equal(full[0, [1, 4, 6]], lg[0])


# --------------------------------------------------------------------- e4m3


def test_e4m3_rounding_against_torch_and_tie_cases():
    import torch

    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(2000) * 1e-2,
                        np.linspace(-448, 448, 4001)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(ref.e4m3_round(x), want)
    # ties to even and saturation
    cases = {1.0625: 1.0, 1.1875: 1.25, 2.0**-10: 0.0, 3 * 2.0**-10: 2.0**-8, 500.0: 448.0, -1e6: -448.0}
    for a, b in cases.items():
        assert ref.e4m3_round(np.float32(a)) == b


def test_e4m3_per_channel_scale():
    rng = np.random.default_rng(12)
    w = rng.standard_normal((6, 40)).astype(np.float32)
    w[3] = 0
    q, s = ref.quantize_e4m3_per_channel(w)
    assert s[3] == 1.0 and np.all(q[3] == 0)
    assert np.all(np.max(np.abs(q[[0, 1, 2, 4, 5]]), axis=1) == 448.0)
    deq = ref.dequantize(q, s)
    assert np.max(np.abs(deq - w)) <= np.max(np.abs(w)) / 448 * 16  # half an e4m3 step at the top


def test_e4m3_weight_set_matches_the_pages_list():
    """flashmap/sglang/model.py, _quantize_fp8 lists x_embed, fc, the context/anchor
    projections, the folded head and every block's linears; norms, AdaLN weights and
    the noise factor stay unquantized. The set is fixed by name here, independently of
    the oracle's list."""
    cfg = ref.Config.from_dict(syn.model_config("small_bf16"))
    names = set(ref.e4m3_linear_names(cfg))
    shapes = syn.weight_shapes(syn.model_config("small_bf16"))
    want = {"x_embed.weight", "fc.weight", "anchor_proj.weight"}
    for l in range(cfg.num_layers):
        for att in ("self_attn", "cross_attn"):
            want |= {f"layers.{l}.{att}.{p}_proj.weight" for p in "qkvo"}
        want |= {f"layers.{l}.mlp.fc1.weight", f"layers.{l}.mlp.fc2.weight"}
    assert names == want
    assert names <= set(shapes)
    assert not any("norm" in n or "adaln" in n or "embed." in n.replace("x_embed", "") for n in names)


def test_e4m3_weights_quantize_only_the_set_and_stay_within_half_a_step():
    cfg = ref.Config.from_dict(syn.model_config("tiny_fp32"))
    rng = np.random.default_rng(5)
    W = {n: rng.standard_normal(s).astype(np.float32) for n, s in syn.weight_shapes(syn.model_config("tiny_fp32")).items()}
    Wq = ref.e4m3_weights(cfg, W)
    qset = set(ref.e4m3_linear_names(cfg))
    for n, w in W.items():
        if n not in qset:
            assert Wq[n] is w
            continue
        amax = np.max(np.abs(w), axis=1, keepdims=True)
        scale = amax / 448.0
        # every dequantized value is an e4m3 value times its row's scale ...
        q = Wq[n] / scale.astype(np.float32).astype(np.float64)
        np.testing.assert_array_equal(ref.e4m3_round(q.astype(np.float32)), q)
        # ... within half an e4m3 step (relative 2^-4) of the original, or 2^-10 scale absolute
        err = np.abs(Wq[n] - w)
        assert np.all(err <= np.maximum(np.abs(w) * 2.0**-4, scale * 2.0**-10) * (1 + 1e-6))
        # the row maximum maps to exactly 448 * scale
        np.testing.assert_allclose(np.max(np.abs(Wq[n]), axis=1), amax[:, 0], rtol=1e-6)


def test_e4m3_constants_quantize_the_folded_head_only():
    cfg = ref.Config.from_dict(syn.model_config("tiny_fp32"))
    rng = np.random.default_rng(6)
    C = ref.Constants(mods=None, final=None, gate=1.0, uniform=None, gram=None, chol=None,
                      hot=np.arange(8), head_w=rng.standard_normal((8, 16)), head_b=rng.standard_normal(8))
    Cq = ref.e4m3_constants(C)
    assert Cq.head_b is C.head_b and Cq.hot is C.hot
    assert not np.array_equal(Cq.head_w, C.head_w)
    assert np.max(np.abs(Cq.head_w - C.head_w)) <= np.max(np.abs(C.head_w)) / 448 * 16


# --------------------------------------------------------------------- verify tree


def _read_tree_golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "tree_example.txt")
    vals = {}
    for ln in open(path):
        ln = ln.strip()
        if ln and not ln.startswith("#"):
            key, *rest = ln.split()
            vals[key] = [int(x) for x in rest]
    return vals


def test_tree_hand_worked_example():
    g = _read_tree_golden()
    c = np.array(g["candidates"]).reshape(g["n"][0], g["k"][0])
    tokens, ids, stats = ref.build_tree(c, g["width"][0])
    np.testing.assert_array_equal(tokens, g["tokens"])
    np.testing.assert_array_equal(ids, g["ids"])
    np.testing.assert_array_equal(stats, g["stats"])


def _decode(tokens, ids, width):
    """Node number -> (parent number, token, path of tokens from the root)."""
    out = {}
    for q, (t, i) in enumerate(zip(tokens, ids)):
        parent, num = divmod(int(i), width)
        assert num == q + 1
        out[num] = (parent, int(t))
    return out


@pytest.mark.parametrize("seed,n,k,width,alphabet", [(0, 8, 4, 16, 3), (1, 16, 6, 40, 2), (2, 4, 3, 64, 5),
                                                     (3, 32, 16, 64, 4), (4, 1, 5, 8, 9)])
def test_tree_invariants_on_random_candidates(seed, n, k, width, alphabet):
    """Every kept node's parent is kept and listed before it; each node's path from the
    root is a prefix of some candidate with exactly as many candidates through it as
    the trie says; no dropped prefix outranks a kept one; padding repeats the first
    node under the root; stats count the trie's nodes and the distinct candidates."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, alphabet, size=(n, k))
    tokens, ids, stats = ref.build_tree(c, width)
    m = width - 1
    assert tokens.shape == (m,) and ids.shape == (m,)
    rows = [tuple(r) for r in c.tolist()]
    prefixes = {}  # prefix -> the candidates through it, with repeats (a vote each)
    for r in rows:
        for d in range(k):
            prefixes.setdefault(r[:d + 1], []).append(r)
    assert stats[0] == len(prefixes) and stats[1] == len(set(rows))
    nodes = _decode(tokens, ids, width)
    kept = min(m, len(prefixes))
    paths = {}
    for num in range(1, kept + 1):
        parent, t = nodes[num]
        assert parent < num
        paths[num] = (paths[parent] if parent else ()) + (t,)
        assert paths[num] in prefixes
    assert len(set(paths.values())) == kept  # distinct nodes
    for num in range(kept + 1, m + 1):  # padding
        assert nodes[num] == (0, nodes[1][1]) and len(paths[1]) == 1
    # the cut: no dropped node has more votes than a kept one (ties: shallower first)
    rank = lambda p: (-len(prefixes[p]), len(p), min(rows.index(r) for r in prefixes[p]))
    kept_ranks = [rank(p) for p in paths.values()]
    dropped = [rank(p) for p in prefixes if p not in set(paths.values())]
    if dropped:
        assert max(kept_ranks) < min(dropped)
    # listing order: by depth, then by lowest candidate through the node
    order = [(len(paths[q]), rank(paths[q])[2]) for q in range(1, kept + 1)]
    assert order == sorted(order)


def test_candidate_noise_keying():
    """Reading R7: candidate 0's noise is the single draft's; other candidates draw
    fresh N(0, 1) noise, uncorrelated with candidate 0's, from the same seed."""
    pos = np.arange(100, 164)
    z0 = ref.draft_normals(12345, pos, 256)
    np.testing.assert_array_equal(ref.draft_normals(12345, pos, 256, candidate=0), z0)
    z3 = ref.draft_normals(12345, pos, 256, candidate=3)
    assert not np.allclose(z3, z0)
    assert st.kstest(z3.reshape(-1), "norm").pvalue > 1e-3
    assert abs(np.corrcoef(z0.reshape(-1), z3.reshape(-1))[0, 1]) < 0.02


# --------------------------------------------------------------------- several jumps


def test_embed_state_at_zero_is_the_cholesky_path(tiny):
    """At s = 0 the posterior is uniform whatever the state, and the state enters only
    as x0 @ E: with z solving z L^T = x0 @ E, embed_state equals the one-jump
    embedding u + gate * noise_norm(z L^T) (modeling_flashmap.py, target_constants)."""
    cfg, W, E, LM, rank, C = tiny
    rng = np.random.default_rng(3)
    x0 = rng.standard_normal((6, cfg.vocab_size))
    z = np.linalg.solve(C.chol, (x0 @ E.astype(np.float64)).T).T
    np.testing.assert_allclose(ref.embed_state(cfg, W, C, E, x0, 0.0, 1.0), ref.embed_noise(cfg, W, C, z),
                               rtol=1e-9, atol=1e-9)
    # with a zero jump (gate 0) only the posterior term is left: the uniform constant
    # at s = 0 whatever the state, a function of the state for s > 0
    np.testing.assert_allclose(ref.embed_state(cfg, W, C, E, x0, 0.0, 0.0),
                               np.broadcast_to(C.uniform, (6, C.uniform.shape[0])), rtol=1e-12)
    b = ref.embed_state(cfg, W, C, E, x0, 0.5, 0.5) - ref.embed_state(cfg, W, C, E, 2 * x0, 0.5, 0.5)
    assert not np.allclose(b, 0.0, atol=1e-6)


def test_jump_state_update_and_grid():
    """The state recurrence of the jump loop: with t - s the weight of the DiT's
    distribution, a state already equal to that distribution is a fixed point, and the
    printed grids start at 0 and end at 1 with increasing times."""
    for n, grid in ref.DEFAULT_JUMP_GRIDS.items():
        assert grid[0] == 0.0 and grid[-1] == 1.0 and len(grid) == int(n) + 1
        assert all(a < b for a, b in zip(grid[:-1], grid[1:]))
    # on the interpolant x_s = (1 - s) x0 + s x1 of the flow, a jump s -> t toward
    # x1 lands on x_t = (1 - t) x0 + t x1, over every printed grid in turn
    rng = np.random.default_rng(4)
    x0 = rng.standard_normal((3, 50))
    x1 = ref.softmax(rng.standard_normal((3, 50)))
    for grid in ref.DEFAULT_JUMP_GRIDS.values():
        x = x0.copy()
        for s, t in zip(grid[:-1], grid[1:]):
            np.testing.assert_allclose(x, (1 - s) * x0 + s * x1, rtol=1e-9, atol=1e-12)
            x = ref.jump_state(x, x1, s, t)
        np.testing.assert_allclose(x, x1, rtol=1e-9, atol=1e-12)


def test_state_posterior_is_the_gaussian_bayes_posterior():
    """At time s the state of token j is distributed N(s e_j, (1 - s)^2 I); with a
    uniform prior, Bayes' rule over the V candidates gives the posterior the jump
    embeds. Brute force with scipy's Gaussian log-density on a small vocabulary."""
    from scipy.stats import multivariate_normal

    rng = np.random.default_rng(5)
    V = 7
    for s in (0.2, 0.5, 0.8172569274902344):
        j_true = 3
        x = (1 - s) * rng.standard_normal(V) + s * np.eye(V)[j_true]
        logp = np.array([multivariate_normal.logpdf(x, mean=s * np.eye(V)[j], cov=(1 - s) ** 2 * np.eye(V))
                         for j in range(V)])
        bayes = np.exp(logp - logp.max())
        bayes /= bayes.sum()
        np.testing.assert_allclose(ref.state_posterior(x[None], s)[0], bayes, rtol=1e-9)
    # at s = 0 the posterior is uniform
    np.testing.assert_allclose(ref.state_posterior(rng.standard_normal((2, V)), 0.0), np.full((2, V), 1 / V))


# --------------------------------------------------------------------- folded-noise eigenbasis


def test_noise_basis_closed_form_2x2():
    """A 2 x 2 gram [[a, b], [b, c]]: eigenvalues (a + c)/2 -/+ sqrt(((a - c)/2)^2 + b^2)
    and the eigenvector of lam along (b, lam - a), signed by reading R9."""
    for a, b, c in ((2.0, 0.7, 1.0), (1.0, -0.3, 3.0), (0.5, 0.2, 0.5)):
        lam, Q = ref.noise_basis(np.array([[a, b], [b, c]]))
        half, rad = (a + c) / 2, math.hypot((a - c) / 2, b)
        np.testing.assert_allclose(lam, [half - rad, half + rad], rtol=1e-13)
        for i, l in enumerate((half - rad, half + rad)):
            v = np.array([b, l - a])
            v /= np.linalg.norm(v)
            v *= 1.0 if v[np.argmax(np.abs(v))] > 0 else -1.0
            np.testing.assert_allclose(Q[:, i], v, rtol=1e-12, atol=1e-14)


def test_noise_basis_reconstructs_the_gram(tiny):
    cfg, W, E, LM, rank, C = tiny
    lam, Q = ref.noise_basis(C.gram)
    G = E.astype(np.float64).T @ E.astype(np.float64)
    assert np.linalg.norm((Q * lam) @ Q.T - G) / np.linalg.norm(G) < 1e-12
    np.testing.assert_allclose(Q.T @ Q, np.eye(G.shape[0]), atol=1e-12)
    assert np.all(np.diff(lam) >= 0) and np.all(lam >= 0)
    lead = Q[np.argmax(np.abs(Q), axis=0), np.arange(Q.shape[1])]
    assert np.all(lead > 0)


def test_folded_noise_is_the_unfolded_embedding():
    """flashmap/sglang/model.py, _folded_noise: x_embed(u + gate * noise_norm(y)) with
    y = (z * sqrt(lam)) @ Q^T equals x_embed(u) + gate * r * (z @ M), the unfolded side
    written with the pinned rms_norm and a plain x_embed; a gate != 1 and a noise norm
    weight far from 1 make a dropped factor fail."""
    cfg, W, E, LM, rank = _tiny(noise_path=1)
    W = dict(W)
    rng = np.random.default_rng(8)
    W["noise_norm.weight"] = (1.0 + 0.5 * rng.standard_normal(cfg.target_hidden)).astype(np.float32)
    W["noise_gate"] = np.array([0.7], dtype=np.float32)
    C = ref.load_constants(cfg, W, E, LM, rank)
    F = C.extra["folded"]
    lam, Q = ref.noise_basis(C.gram)
    z = rng.standard_normal((5, cfg.target_hidden)) * 1.3
    y = (z * np.sqrt(lam)) @ Q.T
    e = C.uniform + C.gate * ref.rms_norm(y, W["noise_norm.weight"], cfg.rms_norm_eps)
    unfolded = e @ W["x_embed.weight"].astype(np.float64).T + W["x_embed.bias"]
    np.testing.assert_allclose(ref.embed_noise_folded(cfg, F, C.gate, z), unfolded, rtol=1e-10, atol=1e-12)
    # the draft's noise embedding takes this path when noise_path = 1
    x = ref.noise_embedding(cfg, W, C, 17, np.arange(3, 3 + cfg.block_size), 1.0)
    z2 = ref.draft_normals(17, np.arange(3, 3 + cfg.block_size), cfg.target_hidden)
    np.testing.assert_allclose(x, ref.embed_noise_folded(cfg, F, C.gate, z2), rtol=1e-13)


def test_folded_noise_law_matches_embedding_covariance():
    """(z * sqrt(lam)) @ Q^T ~ N(0, E^T E), like z L^T; a transposed basis (Q diag(lam)
    read as rows) fails on a gram far from a multiple of the identity."""
    rng = np.random.default_rng(9)
    V, H, N = 512, 24, 60000
    E = rng.standard_normal((V, H)) @ (rng.standard_normal((H, H)) + 2 * np.eye(H)) * 0.05
    G = E.T @ E
    lam, Q = ref.noise_basis(G)
    z = ref.draft_normals(7, np.arange(N), H)
    y = (z * np.sqrt(lam)) @ Q.T
    assert np.linalg.norm(y.T @ y / N - G) / np.linalg.norm(G) < 0.05
    wrong = (z * np.sqrt(lam)) @ Q
    assert np.linalg.norm(wrong.T @ wrong / N - G) / np.linalg.norm(G) > 0.2


# --------------------------------------------------------------------- DiT wiring
#
# modeling_flashmap.py, FlashMapAdaLayerNorm.modulation / forward, FlashMapLayer.forward,
# FlashMapDraftModel.time_conditioning and draft fix which modulation chunk is the scale,
# the shift and the gate, which branch each AdaLN feeds, that time_embed reads the jump's
# start s and jump_embed its end t, and where the block's slots sit (anchor + 1 + k).
# Every expected value below is built from scipy routines or from the pinned primitives
# (rms_norm, apply_rope, attention, time_embedding); a swapped chunk, branch, time or
# position fails one of them.


def _zero_adaln(W, cfg, biases):
    """Zero every AdaLN weight and set its bias: biases[name] = (scale, shift, gate)
    vectors (missing names: all zero). Returns the modified copy of W."""
    W = dict(W)
    D = cfg.hidden
    names = [f"layers.{l}.{n}" for l in range(cfg.num_layers)
             for n in ("self_attn_adaln", "cross_attn_adaln", "mlp_adaln")] + ["final_adaln"]
    for n in names:
        W[f"{n}.linear.weight"] = np.zeros((3 * D, cfg.cond_dim))
        sc, sh, g = biases.get(n, (np.zeros(D), np.zeros(D), np.zeros(D)))
        W[f"{n}.linear.bias"] = np.concatenate([sc, sh, g])
    return W


def test_adaln_chunks_are_scale_shift_gate():
    """FlashMapAdaLayerNorm.modulation returns (scale, shift, gate), used as
    norm(x) * (1 + scale) + shift with gate on the residual: zero weights and distinct
    bias chunks must come back as (1 + b_scale, b_shift, b_gate) per norm, in the
    order (self-attention, cross-attention, MLP), and (1 + b_scale, b_shift) for the
    final norm."""
    cfg, W, E, LM, rank = _tiny()
    rng = np.random.default_rng(40)
    D = cfg.hidden
    biases = {}
    for l in range(cfg.num_layers):
        for j, n in enumerate(("self_attn_adaln", "cross_attn_adaln", "mlp_adaln")):
            biases[f"layers.{l}.{n}"] = tuple(rng.standard_normal(D) + 10 * (9 * l + 3 * j + c) for c in range(3))
    biases["final_adaln"] = tuple(rng.standard_normal(D) - 10 * (c + 1) for c in range(3))
    W = _zero_adaln(W, cfg, biases)
    mods, final, _ = ref.jump_conditioning(cfg, W, 0.0, 1.0)
    for l in range(cfg.num_layers):
        for j, n in enumerate(("self_attn_adaln", "cross_attn_adaln", "mlp_adaln")):
            sc, sh, g = biases[f"layers.{l}.{n}"]
            np.testing.assert_array_equal(mods[l, 3 * j + 0], 1.0 + sc)
            np.testing.assert_array_equal(mods[l, 3 * j + 1], sh)
            np.testing.assert_array_equal(mods[l, 3 * j + 2], g)
    sc, sh, _ = biases["final_adaln"]
    np.testing.assert_array_equal(final[0], 1.0 + sc)
    np.testing.assert_array_equal(final[1], sh)


def _te(W, name, t, cfg):
    return ref.time_embedding(t, W[f"{name}.linear_1.weight"], W[f"{name}.linear_1.bias"],
                              W[f"{name}.linear_2.weight"], W[f"{name}.linear_2.bias"],
                              cfg.time_embed_dim, cfg.time_scale)


@pytest.mark.parametrize("s,t", [(0.0, 1.0), (0.8172569274902344, 1.0), (0.7906050682067871, 0.8172569274902344)])
def test_time_conditioning_reads_s_in_time_embed_and_t_in_jump_embed(s, t):
    """time_conditioning: cond = time_embed(s) + jump_embed(t). With time_embed's
    output layer zeroed, cond is jump_embed at t (not at s); with jump_embed's zeroed,
    time_embed at s (not at t)."""
    cfg, W, E, LM, rank = _tiny()
    H1 = cfg.cond_dim
    zero_te = dict(W, **{"time_embed.linear_2.weight": np.zeros((H1, H1)), "time_embed.linear_2.bias": np.zeros(H1)})
    _, _, cond = ref.jump_conditioning(cfg, zero_te, s, t)
    np.testing.assert_allclose(cond, _te(W, "jump_embed", t, cfg), rtol=1e-13, atol=1e-15)
    assert np.max(np.abs(cond - _te(W, "jump_embed", s, cfg))) > 1e-3  # the test can tell s from t
    zero_je = dict(W, **{"jump_embed.linear_2.weight": np.zeros((H1, H1)), "jump_embed.linear_2.bias": np.zeros(H1)})
    _, _, cond = ref.jump_conditioning(cfg, zero_je, s, t)
    np.testing.assert_allclose(cond, _te(W, "time_embed", s, cfg), rtol=1e-13, atol=1e-15)
    assert np.max(np.abs(cond - _te(W, "time_embed", t, cfg))) > 1e-3


def _layer_case(seed, **over):
    """The tiny model with one DiT layer and layer_norm_eps 0 (so that LayerNorm is
    scipy's z-score), a block x of K slots and a random rotated context."""
    cfg, W, E, LM, rank = _tiny(num_layers=1, layer_norm_eps=0.0, **over)
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((cfg.block_size, cfg.hidden)) * 2 + 0.5
    return cfg, W, rng, x


def _mods_from(W, cfg):
    return ref.jump_conditioning(cfg, W, 0.0, 1.0)[0][0]


def test_mlp_branch_wiring():
    """FlashMapLayer.forward's last branch with the two attention gates zero:
    x + gate * fc2(gelu(fc1(z(x) * (1 + scale) + shift))). fc1 = [I; 0] and
    fc2 = [I, 0] with zero biases make the MLP gelu(h) = h * Phi(h) (scipy), so a
    swapped scale/shift, a missing (1 + .) or a gate on the wrong chunk fails."""
    cfg, W, rng, x = _layer_case(41)
    D, F = cfg.hidden, cfg.intermediate
    sc, sh, g = rng.standard_normal(D) * 0.5, rng.standard_normal(D), rng.standard_normal(D)
    W = _zero_adaln(W, cfg, {"layers.0.mlp_adaln": (sc, sh, g)})  # attention gates 0
    W["layers.0.mlp.fc1.weight"] = np.eye(F, D)
    W["layers.0.mlp.fc1.bias"] = np.zeros(F)
    W["layers.0.mlp.fc2.weight"] = np.eye(D, F)
    W["layers.0.mlp.fc2.bias"] = np.zeros(D)
    p = 6
    ctx = [(rng.standard_normal((p + 1, cfg.num_heads, cfg.head_dim)),) * 2]
    out = ref.dit_layer(cfg, W, 0, _mods_from(W, cfg), x, p + 1 + np.arange(cfg.block_size), ctx)
    h = st.zscore(x, axis=-1) * (1.0 + sc) + sh
    np.testing.assert_allclose(out, x + g * (h * st.norm.cdf(h)), rtol=1e-11, atol=1e-12)


def test_cross_attention_wiring_one_position_context():
    """With every gate but the cross-attention's zero and a context of one position,
    the layer adds gate * (v W_o^T) to every slot whatever its query: the softmax over
    one key is 1 (FlashMapLayer.forward, FlashMapAttention.forward)."""
    cfg, W, rng, x = _layer_case(42)
    D = cfg.hidden
    g = rng.standard_normal(D)
    W = _zero_adaln(W, cfg, {"layers.0.cross_attn_adaln": (rng.standard_normal(D), rng.standard_normal(D), g)})
    k1 = rng.standard_normal((1, cfg.num_heads, cfg.head_dim))
    v1 = rng.standard_normal((1, cfg.num_heads, cfg.head_dim))
    out = ref.dit_layer(cfg, W, 0, _mods_from(W, cfg), x, 1 + np.arange(cfg.block_size), [(k1, v1)])
    want = x + g * (v1.reshape(1, D) @ np.asarray(W["layers.0.cross_attn.o_proj.weight"], np.float64).T)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def test_self_attention_wiring_uniform_scores_average_the_whole_block():
    """With q_proj = 0 the normed queries are 0, every score is 0 and the attention
    averages the values of all K slots of the block, the later ones included (the
    block attends non-causally). Only the self-attention gate is nonzero: the layer
    adds gate * mean_k(v_k) W_o^T, v = W_v (z(x) * (1 + scale) + shift); a causal mask
    (prefix means) or the shift/scale swapped fails."""
    cfg, W, rng, x = _layer_case(43)
    D = cfg.hidden
    sc, sh, g = rng.standard_normal(D) * 0.5, rng.standard_normal(D), rng.standard_normal(D)
    W = _zero_adaln(W, cfg, {"layers.0.self_attn_adaln": (sc, sh, g)})
    W["layers.0.self_attn.q_proj.weight"] = np.zeros((D, D))
    p = 3
    ctx = [(rng.standard_normal((p + 1, cfg.num_heads, cfg.head_dim)),) * 2]
    out = ref.dit_layer(cfg, W, 0, _mods_from(W, cfg), x, p + 1 + np.arange(cfg.block_size), ctx)
    h = st.zscore(x, axis=-1) * (1.0 + sc) + sh
    v = h @ np.asarray(W["layers.0.self_attn.v_proj.weight"], np.float64).T
    o = np.asarray(W["layers.0.self_attn.o_proj.weight"], np.float64)
    want = x + g * (v.mean(axis=0, keepdims=True) @ o.T)
    np.testing.assert_allclose(out, want, rtol=1e-11, atol=1e-12)


def test_layer_is_equivariant_to_permuting_slots_with_their_positions():
    """Non-causal self-attention and row-wise everything else: permuting a request's
    slots together with their positions permutes the layer's output rows (all weights
    random, every gate nonzero). A causal mask or a position taken from the row index
    instead of the given position fails."""
    cfg, W, rng, x = _layer_case(44)
    p = 9
    pos = p + 1 + np.arange(cfg.block_size)
    kc = rng.standard_normal((p + 1, cfg.num_heads, cfg.head_dim))
    vc = rng.standard_normal((p + 1, cfg.num_heads, cfg.head_dim))
    mods = _mods_from(W, cfg)
    out = ref.dit_layer(cfg, W, 0, mods, x, pos, [(kc, vc)])
    perm = np.array([2, 0, 3, 1])
    out_p = ref.dit_layer(cfg, W, 0, mods, x[perm], pos[perm], [(kc, vc)])
    np.testing.assert_allclose(out_p, out[perm], rtol=1e-12, atol=1e-12)
    # a permutation of the rows that keeps the positions in place changes the result
    out_q = ref.dit_layer(cfg, W, 0, mods, x[perm], pos, [(kc, vc)])
    assert np.max(np.abs(out_q - out[perm])) > 1e-4


def _context_at(cfg, W, E, hid, anchor, start):
    """Every layer's rotated context for target hidden states at positions start ..
    start+p-1 and the anchor at start+p (write_rows_kv, anchor_kv)."""
    p = hid.shape[0]
    kw, vw = ref.write_rows_kv(cfg, W, hid, start + np.arange(p))
    ka, va = ref.anchor_kv(cfg, W, E, anchor, [start + p])
    return np.concatenate([kw, ka], axis=1), np.concatenate([vw, va], axis=1)


def test_draft_is_invariant_to_shifting_every_position():
    """RoPE makes every attention score a function of position differences, so at
    noise_scale 0 (no position-keyed noise) moving a whole request by delta -- context
    at delta..delta+p-1, anchor at delta+p, slots from delta+p+1 -- leaves every
    layer's output unchanged up to the float32 angles. Queries rotated at other
    positions than the keys (here: left unshifted) fail."""
    cfg, W, E, LM, rank = _tiny(num_layers=2)
    C = ref.load_constants(cfg, W, E, LM, rank)
    rng = np.random.default_rng(45)
    p, K = 12, cfg.block_size
    hid = rng.standard_normal((p, cfg.num_target_layers * cfg.target_hidden))
    anchor = [int(rng.integers(cfg.vocab_size))]

    def layers(start, slot_start):
        kc, vc = _context_at(cfg, W, E, hid, anchor, start)
        pos = slot_start + np.arange(K)
        x = ref.noise_embedding(cfg, W, C, 5, pos, 0.0)
        for l in range(cfg.num_layers):
            x = ref.dit_layer(cfg, W, l, C.mods[l], x, pos, [(kc[l], vc[l])])
        return x

    base = layers(0, p + 1)
    np.testing.assert_allclose(layers(7, p + 8), base, rtol=0, atol=2e-5 * np.max(np.abs(base)))
    np.testing.assert_allclose(layers(300, p + 301), base, rtol=0, atol=2e-4 * np.max(np.abs(base)))
    assert np.max(np.abs(layers(7, p + 1) - base)) > 1e-2 * np.max(np.abs(base))  # the test can tell


def test_slots_sit_after_the_anchor():
    """modeling_flashmap.py, draft: the block's slots are at anchor + 1 + k and attend
    to the context 0..anchor. One layer whose only nonzero gate is the cross-attention's
    and whose cross modulation has scale -1 (so 1 + scale = 0) gives every slot the same
    pre-rotation query q = q_norm(W_q shift); the slots then differ only by the
    rotation of q at their positions. At noise_scale 0 and with a final AdaLN of scale 0
    and shift 0, the draft is z(x0 + gate * attention(R_pos q, K, V) W_o^T), built here
    from the pinned rms_norm, apply_rope and attention. Slots at anchor + k fail."""
    cfg, W, E, LM, rank = _tiny(num_layers=1, layer_norm_eps=0.0)
    rng = np.random.default_rng(46)
    D, nh, hd, K = cfg.hidden, cfg.num_heads, cfg.head_dim, cfg.block_size
    shift, g = rng.standard_normal(D), rng.standard_normal(D)
    W = _zero_adaln(W, cfg, {"layers.0.cross_attn_adaln": (-np.ones(D), shift, g)})
    C = ref.load_constants(cfg, W, E, LM, rank)
    p = 5
    kc = rng.standard_normal((1, p + 1, nh, hd)) * 3
    vc = rng.standard_normal((1, p + 1, nh, hd))
    out = ref.draft_requests(cfg, W, C, [(kc, vc)], [p], [9], noise_scale=0.0)[0]

    x0 = ref.noise_embedding(cfg, W, C, 9, p + 1 + np.arange(K), 0.0)
    wq = np.asarray(W["layers.0.cross_attn.q_proj.weight"], np.float64)
    q = ref.rms_norm((shift @ wq.T).reshape(1, nh, hd), W["layers.0.cross_attn.q_norm.weight"], cfg.qk_norm_eps)
    wo = np.asarray(W["layers.0.cross_attn.o_proj.weight"], np.float64)

    def expected(first_slot):
        pos = first_slot + np.arange(K)
        qr = ref.apply_rope(np.repeat(q, K, axis=0), pos, cfg.rope_theta)
        att = ref.attention(qr, kc[0], vc[0]).reshape(K, D)
        return st.zscore(x0 + g * (att @ wo.T), axis=-1)

    np.testing.assert_allclose(out, expected(p + 1), rtol=1e-10, atol=1e-10)
    assert np.max(np.abs(out - expected(p))) > 1e-3  # the test can tell


def test_e4m3_query_quantization_hand_worked():
    """flashmap/sglang/model.py, _paged_cross_attention_fp8: per (request, head) the
    query scale is max(max|q|, 1e-12) / 448 and q8 = e4m3(q / scale). Worked by hand:
    head 0 has max|q| = 448, so its scale is 1 and q8 is q rounded to e4m3 -- 1.0625
    lies halfway between 1 and 1.125 (step 1/8 in [1, 2)) and goes to the even 1.0;
    -3.3 lies in [2, 4) (step 1/4) nearest -3.25; 300 lies in [256, 512) (step 32)
    nearest 288. Head 1's largest magnitude 1e-13 is below the 1e-12 floor: its scale
    is 1e-12 / 448 and 1e-13 / scale = 44.8 lies in [32, 64) (step 4), nearest 44.
    The two slots share one scale per head."""
    q = np.zeros((2, 2, 4))
    q[0, 0] = [448.0, 1.0625, -3.3, 0.0]
    q[1, 0] = [300.0, 0.0, 0.0, 0.0]
    q[0, 1] = [1e-13, -0.5e-13, 0.0, 0.0]
    got = ref.quantize_query_e4m3(q)
    np.testing.assert_array_equal(got[0, 0], [448.0, 1.0, -3.25, 0.0])
    np.testing.assert_array_equal(got[1, 0], [288.0, 0.0, 0.0, 0.0])
    s1 = float(np.float32(np.float32(1e-12) / np.float32(448.0)))
    # -0.5e-13 / s1 = -22.4: [16, 32) has step 2, nearest -22
    np.testing.assert_allclose(got[0, 1], [44.0 * s1, -22.0 * s1, 0.0, 0.0], rtol=1e-6)
