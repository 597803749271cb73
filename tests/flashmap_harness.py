"""Test harness: runs one draft step of a synthetic workload through the C ABI on the
GPU and through the CPU oracle on the same seeded inputs, and compares them.

The oracle never sees a value the CUDA path computed: its inputs are the seeded
draws of ``synthetic`` (weights, hidden states, and, for prefilled workloads, the
N(0, 1) context keys/values that torch wrote into the pool before any library call).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from oracle import flashmap_ref as ref
from speculative_decoding_block_context_gb300 import _lib as F
from speculative_decoding_block_context_gb300 import synthetic as syn

TOL = {"f32": 1e-4, "bf16": 2e-2}
TOKEN_MARGIN = 1e-2


def max_rel(a, b) -> float:
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    den = max(float(np.max(np.abs(b))), 1e-30)
    return float(np.max(np.abs(a - b))) / den


@dataclass
class ModelState:
    cfg: dict
    W: dict  # torch, device
    E: torch.Tensor
    LM: torch.Tensor
    rank: torch.Tensor
    handle: object = None
    Wnp: dict = field(default_factory=dict)  # float32 numpy copies for the oracle
    Enp: np.ndarray = None
    LMnp: np.ndarray = None
    consts: object = None

    def oracle_cfg(self):
        return ref.Config.from_dict(self.cfg)


def load_model(workload: str, device="cuda", oracle: bool = True) -> ModelState:
    cfg = syn.model_config(workload)
    W, E, LM, rank = syn.make_model(cfg, device)
    st = ModelState(cfg, W, E, LM, rank)
    st.handle = F.flashmap_load_weights(cfg, W, E, LM, rank)
    torch.cuda.synchronize()
    if oracle:
        st.Wnp = {k: v.float().cpu().numpy() for k, v in W.items()}
        st.Enp = E.float().cpu().numpy()
        if cfg["weight_dtype"] == "e4m3":  # the oracle runs on the dequantized weights
            st.Wnp = ref.e4m3_weights(st.oracle_cfg(), st.Wnp)
        st.LMnp = LM.float().cpu().numpy()
        st.consts = ref.load_constants(st.oracle_cfg(), st.Wnp, st.Enp, st.LMnp, rank.cpu().numpy())
        if cfg["weight_dtype"] == "e4m3":
            st.consts = ref.e4m3_constants(st.consts)
    return st


def value_byte(cfg: dict) -> torch.Tensor:
    """Where each position of a page sits in an e4m3 pool's channel-major value rows:
    within every 16 positions, position 2t + e at byte 4t + e and position 8 + 2t + e at
    byte 4t + 2 + e (t < 4, e < 2); the identity for other pools."""
    p = torch.arange(cfg["page_size"])
    if cfg["kv_dtype"] != "e4m3":
        return p
    o = p % 16
    return p - o + 4 * ((o % 8) // 2) + 2 * (o // 8) + o % 2


def pool_view(cfg: dict, pool_t: torch.Tensor, num_pages: int) -> tuple:
    """Views of the pool's keys and values as stored: keys (L, pages, heads, P, hd); values
    the same for a bf16 or f32 pool, and for an e4m3 pool, which keeps each (page, head)
    block of values channel-major (hd, P) with the positions in value_byte order, a
    transposed view (L, pages, heads, P, hd) indexed by byte. No copy."""
    dt = syn.torch_dtype(cfg["kv_dtype"])
    L, nh, P, hd = cfg["num_layers"], cfg["num_heads"], cfg["page_size"], cfg["head_dim"]
    kv = pool_t.view(dt).view(L, 2, num_pages * nh * P * hd)
    k = kv[:, 0].view(L, num_pages, nh, P, hd)
    if cfg["kv_dtype"] == "e4m3":
        v = kv[:, 1].view(L, num_pages, nh, hd, P).transpose(-1, -2)
    else:
        v = kv[:, 1].view(L, num_pages, nh, P, hd)
    return k, v


def slot_rows(cfg: dict, kv: tuple, s: torch.Tensor) -> tuple:
    """The (L, n, heads, hd) keys and values at pool slots s (a device int64 tensor)."""
    P = cfg["page_size"]
    vb = value_byte(cfg).to(s.device)
    k, v = kv
    return (k.permute(1, 3, 0, 2, 4)[s // P, s % P].permute(1, 0, 2, 3),
            v.permute(1, 3, 0, 2, 4)[s // P, vb[s % P]].permute(1, 0, 2, 3))


def gather_context(cfg: dict, kv: tuple, req_to_page_row: torch.Tensor, n: int):
    """Keys and values of positions 0..n-1 of one request, read through its page-table
    row: numpy (L, n, heads, hd) x 2."""
    P = cfg["page_size"]
    npages = (n + P - 1) // P
    pages = req_to_page_row[:npages].long()
    vb = value_byte(cfg).to(pages.device)
    out = []
    for i, t in enumerate(kv):
        g = t[:, pages]
        if i == 1:
            g = g[:, :, :, vb]  # positions in order
        g = g.permute(0, 1, 3, 2, 4).reshape(cfg["num_layers"], npages * P, cfg["num_heads"], cfg["head_dim"])
        out.append(g[:, :n].float().cpu().numpy())
    return out[0], out[1]


@dataclass
class LibRun:
    req: dict
    pool_t: torch.Tensor
    prefill_loc: list
    window_loc: torch.Tensor
    anchor_loc: torch.Tensor
    hidden: torch.Tensor
    tokens: torch.Tensor
    logits: torch.Tensor
    full: torch.Tensor
    prefilled_ctx: dict  # b -> (K, V) numpy of the drawn context (prefilled workloads)
    dev_err: int
    cfg: dict

    @property
    def kv(self) -> tuple:
        """Views of the pool's keys and values (see pool_view)."""
        return pool_view(self.cfg, self.pool_t, self.req["num_pages"])


def run_library(workload: str, st: ModelState, *, noise_scale: float = 1.0, check_subset=None,
                req: dict | None = None, deferred: bool = False) -> LibRun:
    """One step through the C ABI. deferred: the verify-window write goes to
    flashmap_draft_block_with_write instead of its own flashmap_write_context_kv call."""
    cfg, dev = st.cfg, "cuda"
    req = req or syn.make_requests(workload, dev)
    bs, K, D = req["bs"], cfg["block_size"], cfg["hidden"]
    dt = syn.torch_dtype(cfg["act_dtype"])
    code = F.DTYPE_CODES[cfg["kv_dtype"]]
    pool_t = torch.empty(F.flashmap_pool_bytes(cfg, req["num_pages"]), dtype=torch.uint8, device=dev)
    prefilled = {}
    if not req["prefill"]:
        syn.fill_pool_random(pool_t.view(syn.torch_dtype(cfg["kv_dtype"])), req["kv_generator_seed"])
        kv = pool_view(cfg, pool_t, req["num_pages"])
        for b in (check_subset or []):
            row = req["req_to_page"][int(req["req_pool_idx"][b])]
            prefilled[b] = gather_context(cfg, kv, row, req["ctx"][b])
    pool = F.make_pool(pool_t, req["num_pages"], code)
    max_rows = max(max(req["ctx"]) if req["prefill"] else 0, bs * (K + 1))
    ws = torch.empty(F.flashmap_workspace_size(st.handle, bs, min(max_rows, 4096)), dtype=torch.uint8, device=dev)
    prefill_loc = []
    i32 = dict(dtype=torch.int32, device=dev)
    if req["prefill"]:
        for b in range(bs):
            X = req["prefill_hidden"][b]
            n = X.shape[0]
            loc = torch.empty(n, dtype=torch.int64, device=dev)
            F.flashmap_write_context_kv(st.handle, pool, X, 1, n, req["req_pool_idx"][b : b + 1],
                                        torch.zeros(1, **i32), None, req["req_to_page"], loc, ws)
            prefill_loc.append(loc)
    window_loc = None
    anchor_pos = torch.tensor(req["anchor_pos"], **i32)
    hidden = torch.empty((bs * K, D), dtype=dt, device=dev)
    anchor_loc = torch.empty(bs, dtype=torch.int64, device=dev)
    if req["window"]:
        W = K + 1
        window_loc = torch.empty(bs * W, dtype=torch.int64, device=dev)
        start, commit = torch.tensor(req["ctx"], **i32), torch.tensor(req["commit"], **i32)
    if req["window"] and deferred:
        F.flashmap_draft_block_with_write(st.handle, pool, req["window_hidden"], W, start, commit, window_loc, bs,
                                          req["anchor_ids"], anchor_pos, req["req_pool_idx"], req["req_to_page"],
                                          req["seeds"], noise_scale, hidden, anchor_loc, ws)
    else:
        if req["window"]:
            F.flashmap_write_context_kv(st.handle, pool, req["window_hidden"], bs, W, req["req_pool_idx"], start,
                                        commit, req["req_to_page"], window_loc, ws)
        F.flashmap_draft_block(st.handle, pool, bs, req["anchor_ids"], anchor_pos, req["req_pool_idx"],
                               req["req_to_page"], req["seeds"], noise_scale, hidden, anchor_loc, ws)
    Vd = st.consts.hot.shape[0] if st.consts is not None else cfg["draft_vocab_size"] or cfg["vocab_size"]
    tokens = torch.empty(bs * K, dtype=torch.int64, device=dev)
    logits = torch.empty((bs * K, Vd), dtype=torch.float32, device=dev)
    full = (torch.empty((bs * K, cfg["vocab_size"]), dtype=torch.float32, device=dev)
            if req["full_scatter"] else None)
    F.flashmap_sample_block(st.handle, bs, hidden, anchor_pos, req["temperature"], req["greedy"], req["seeds"],
                            req["step"], tokens, logits, full, ws)
    torch.cuda.synchronize()
    err = F.flashmap_get_device_error(st.handle)
    return LibRun(req, pool_t, prefill_loc, window_loc, anchor_loc, hidden, tokens, logits, full,
                  prefilled, err, cfg)


def oracle_batch(st: ModelState, run: LibRun, subset, noise_scale: float = 1.0) -> dict:
    """The oracle's results for the requests in ``subset`` of the run's inputs."""
    cfg, req = st.oracle_cfg(), run.req
    W, C = st.Wnp, st.consts
    K = cfg.block_size
    outs, ctxs, ps, seeds = oracle_contexts(st, run, subset)
    if cfg.num_steps > 1:
        hidden = ref.draft_requests_multi(cfg, W, C, st.Enp, st.LMnp, ctxs, ps, seeds, cfg.num_steps, noise_scale)
    else:
        hidden = ref.draft_requests(cfg, W, C, ctxs, ps, seeds, noise_scale)
    for i, b in enumerate(subset):
        logits = ref.head_logits(C, hidden[i])
        T = float(req["temperature"][b])
        g = int(req["greedy"][b])
        p = ps[i]
        tok, _, margin = ref.sample_rows(logits, [T] * K, [g] * K, [seeds[i]] * K, p + 1 + np.arange(K),
                                         req["step"], C.hot)
        outs[b].update(hidden=hidden[i], logits=logits, tokens=tok, margin=margin)
    return outs


def oracle_contexts(st: ModelState, run: LibRun, subset):
    """Per request of ``subset``: the oracle's written rows (dict), its cross-attention
    context (keys, values over positions 0..p as the pool stores them), p and seed."""
    cfg, req = st.oracle_cfg(), run.req
    W = st.Wnp
    outs, ctxs, ps, seeds = {}, [], [], []
    for b in subset:
        ctx = req["ctx"][b]
        out = {}
        # rows the step writes, as computed (compared with the pool) and as the pool
        # stores them (what the cross-attention reads: e4m3 for an e4m3 pool)
        if req["prefill"]:
            X = req["prefill_hidden"][b].float().cpu().numpy()
            kc, vc = ref.write_rows_kv(cfg, W, X, np.arange(ctx))
            out["prefill_kv"] = (kc, vc)
            kc, vc = ref.store_kv(cfg, kc, vc)
        else:
            kc, vc = run.prefilled_ctx[b]
        if req["window"]:
            m = req["commit"][b]
            X = req["window_hidden"][b, :m].float().cpu().numpy()
            kw, vw = ref.write_rows_kv(cfg, W, X, ctx + np.arange(m))
            out["window_kv"] = (kw, vw)
            kw, vw = ref.store_kv(cfg, kw, vw)
            kc, vc = np.concatenate([kc, kw], axis=1), np.concatenate([vc, vw], axis=1)
        p = req["anchor_pos"][b]
        ka, va = ref.anchor_kv(cfg, W, st.Enp, [int(req["anchor_ids"][b])], [p])
        out["anchor_kv"] = (ka, va)
        ka, va = ref.store_kv(cfg, ka, va)
        ctxs.append((np.concatenate([kc, ka], axis=1), np.concatenate([vc, va], axis=1)))
        ps.append(p)
        seeds.append(int(req["seeds"][b]))
        outs[b] = out
    return outs, ctxs, ps, seeds


def oracle_request(st: ModelState, run: LibRun, b: int, noise_scale: float = 1.0) -> dict:
    return oracle_batch(st, run, [b], noise_scale)[b]


def slot_ids(req: dict, b: int, positions, P: int) -> np.ndarray:
    r2p = req["req_to_page"].cpu().numpy()
    row = int(req["req_pool_idx"][b])
    return np.array([ref.slot_of(r2p, row, int(q), P) for q in positions], dtype=np.int64)


def pool_rows(cfg: dict, kv: tuple, slots) -> tuple:
    """(L, n, heads, hd) keys and values stored at the given slots, numpy."""
    s = torch.as_tensor(np.asarray(slots), device=kv[0].device)
    k, v = slot_rows(cfg, kv, s)
    return k.float().cpu().numpy(), v.float().cpu().numpy()


def kv_err(cfg: dict, got, want, tol: float) -> float:
    """Error of stored keys/values against the oracle's values, on the scale of tol. A
    bf16/f32 pool: max-relative error. An e4m3 pool: every element within half an
    e4m3 step of the oracle's value (2^-4 relative, 2^-10 absolute below the normal
    range) plus tol * max|want|, reported as tol * (worst ratio to that bound)."""
    if cfg.get("kv_dtype") != "e4m3":
        return max_rel(got, want)
    got, want = np.asarray(got, dtype=np.float64), np.asarray(want, dtype=np.float64)
    bound = 2.0**-4 * np.abs(want) + 2.0**-10 + tol * float(np.max(np.abs(want)))
    return tol * float(np.max(np.abs(got - want) / bound))


def check_request(st: ModelState, run: LibRun, b: int, o: dict, tol: float, report: dict) -> None:
    """Compares request b of a library run with the oracle's results ``o``; records the
    worst errors in ``report`` and asserts the bars."""
    cfg, req = st.cfg, run.req
    K, P = cfg["block_size"], cfg["page_size"]
    ctx, p = req["ctx"][b], req["anchor_pos"][b]

    def bump(key, v):
        report[key] = max(report.get(key, 0.0), v)

    if "prefill_kv" in o:
        want = slot_ids(req, b, np.arange(ctx), P)
        got = run.prefill_loc[b].cpu().numpy()
        assert np.array_equal(got, want), "prefill out_loc differs"
        pick = np.unique(np.linspace(0, ctx - 1, min(ctx, 64)).astype(int))
        k, v = pool_rows(cfg, run.kv, want[pick])
        e = max(kv_err(cfg, k, o["prefill_kv"][0][:, pick], tol), kv_err(cfg, v, o["prefill_kv"][1][:, pick], tol))
        bump("write_kv", e)
        assert e <= tol, f"prefill K/V max-rel {e}"
    if "window_kv" in o:
        m = req["commit"][b]
        W = K + 1
        got = run.window_loc.view(-1, W)[b].cpu().numpy()
        want = np.full(W, -1, dtype=np.int64)
        want[:m] = slot_ids(req, b, ctx + np.arange(m), P)
        assert np.array_equal(got, want), "window out_loc differs"
        k, v = pool_rows(cfg, run.kv, want[:m])
        e = max(kv_err(cfg, k, o["window_kv"][0], tol), kv_err(cfg, v, o["window_kv"][1], tol))
        bump("write_kv", e)
        assert e <= tol, f"window K/V max-rel {e}"
    aslot = slot_ids(req, b, [p], P)
    assert int(run.anchor_loc[b]) == int(aslot[0]), "anchor slot differs"
    k, v = pool_rows(cfg, run.kv, aslot)
    e = max(kv_err(cfg, k, o["anchor_kv"][0], tol), kv_err(cfg, v, o["anchor_kv"][1], tol))
    bump("anchor_kv", e)
    assert e <= tol, f"anchor K/V max-rel {e}"
    hid = run.hidden[b * K : (b + 1) * K].float().cpu().numpy()
    e = max_rel(hid, o["hidden"])
    bump("hidden", e)
    assert e <= tol, f"draft hidden max-rel {e}"
    lg = run.logits[b * K : (b + 1) * K].cpu().numpy()
    e = max(max_rel(lg[r], o["logits"][r]) for r in range(K))
    bump("logits", e)
    assert e <= tol, f"logits max-rel {e}"
    tok = run.tokens[b * K : (b + 1) * K].cpu().numpy()
    # A token is decided where the oracle's top-2 margin exceeds 1e-2 and also twice the
    # row's measured logit error (divided by T on sampled rows, whose maximised quantity
    # is l/T + G): within the logits tolerance a smaller margin may flip either way.
    # The report counts the tokens this second condition leaves out
    # (tokens_guarded: margin above 1e-2 but within twice the row's error).
    T, g = float(req["temperature"][b]), int(req["greedy"][b])
    scale = 1.0 if (g or T <= 0.0) else 1.0 / T
    err_row = np.abs(lg - o["logits"]).max(axis=1) * scale
    report["max_token_err"] = max(report.get("max_token_err", 0.0), float(err_row.max()))
    wide = o["margin"] > TOKEN_MARGIN
    sure = wide & (o["margin"] > 2.0 * err_row)
    report["tokens_checked"] = report.get("tokens_checked", 0) + int(sure.sum())
    report["tokens_margin_ok"] = report.get("tokens_margin_ok", 0) + int(wide.sum())
    report["tokens_guarded"] = report.get("tokens_guarded", 0) + int((wide & ~sure).sum())
    report["tokens_total"] = report.get("tokens_total", 0) + K
    if not np.array_equal(tok[sure], o["tokens"][sure]):
        bad = np.nonzero(sure & (tok != o["tokens"]))[0]
        detail = [(int(r), float(o["margin"][r]), float(np.abs(lg[r] - o["logits"][r]).max()),
                   float(np.abs(o["logits"][r]).max())) for r in bad]
        raise AssertionError(f"tokens differ at (slot, oracle margin, max |logit error|, max |logit|) {detail}: "
                             f"{tok} vs {o['tokens']}")


def run_candidates(st: ModelState, run: LibRun, n: int, width: int):
    """Tree drafting on top of a library run (its pool holds every written row): n
    candidate blocks per request (flashmap_draft_candidates), their greedy tokens
    (flashmap_sample_block over bs * n blocks) and the verify trees
    (flashmap_build_tree). Returns (hidden, logits, tokens, (tree tokens, ids, stats))."""
    from speculative_decoding_block_context_gb300 import synthetic as syn

    req, cfg = run.req, st.cfg
    bs, K, D = req["bs"], cfg["block_size"], cfg["hidden"]
    dt = syn.torch_dtype(cfg["act_dtype"])
    pool = F.make_pool(run.pool_t, req["num_pages"], F.DTYPE_CODES[cfg["kv_dtype"]])
    ws = torch.empty(F.flashmap_workspace_size(st.handle, bs * n, bs * (K + 1)), dtype=torch.uint8, device="cuda")
    hidden = torch.empty((bs * n * K, D), dtype=dt, device="cuda")
    anchor_pos = torch.tensor(req["anchor_pos"], dtype=torch.int32, device="cuda")
    F.flashmap_draft_candidates(st.handle, pool, bs, n, req["anchor_ids"], anchor_pos, req["req_pool_idx"],
                                req["req_to_page"], req["seeds"], 1.0, hidden, None, ws)
    rep = lambda t: t.repeat_interleave(n)  # noqa: E731
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
    return hidden, logits, tokens, (t_out, i_out, s_out)


def check_candidates(st: ModelState, run: LibRun, n: int, width: int, tol: float, margin_min: float, subset,
                     out) -> dict:
    """Every candidate block of the requests in ``subset`` against the oracle's draft
    with candidate-keyed noise (hidden states, logits within tol); greedy tokens equal
    wherever the oracle's top-2 margin exceeds margin_min; and every request's tree
    equal, bit for bit, to the oracle's trie over its candidates' tokens -- the oracle's
    token wherever its margin is clear (the library's must be the same there) and the
    library's token at a near tie, where either choice is a valid greedy draw within
    the logits tolerance. Returns counts."""
    hidden, logits, tokens, (t_out, i_out, s_out) = out
    cfg, req = st.cfg, run.req
    bs, K, D = req["bs"], cfg["block_size"], cfg["hidden"]
    vd = st.consts.hot.shape[0]
    h = hidden.float().view(bs, n, K, D)
    _, ctxs, ps, seeds = oracle_contexts(st, run, list(subset))
    blocks = [(i, c) for i in range(len(subset)) for c in range(n)]
    want = ref.draft_requests(st.oracle_cfg(), st.Wnp, st.consts, [ctxs[i] for i, _ in blocks],
                              [ps[i] for i, _ in blocks], [seeds[i] for i, _ in blocks], 1.0, [c for _, c in blocks])
    counts = {"blocks": 0, "tokens": 0, "tokens_clear": 0, "trees": 0, "trees_all_clear": 0}
    for i, b in enumerate(subset):
        mixed = []
        all_clear = True
        for c in range(n):
            hb = h[b, c].cpu().numpy()
            assert max_rel(hb, want[i * n + c]) <= tol, (b, c, max_rel(hb, want[i * n + c]))
            lg = ref.head_logits(st.consts, want[i * n + c])
            got_lg = logits.view(bs, n, K, vd)[b, c].cpu().numpy()
            assert max(max_rel(got_lg[r], lg[r]) for r in range(K)) <= tol
            tok, _, margin = ref.sample_rows(lg, [0.0] * K, [1] * K, [seeds[i]] * K, ps[i] + 1 + np.arange(K), 0,
                                             st.consts.hot)
            got = tokens.view(bs, n, K)[b, c].cpu().numpy()
            sure = margin > margin_min
            np.testing.assert_array_equal(got[sure], tok[sure])
            mixed.append(np.where(sure, tok, got))
            all_clear &= bool(sure.all())
            counts["blocks"] += 1
            counts["tokens"] += K
            counts["tokens_clear"] += int(sure.sum())
        wt, wi, wst = ref.build_tree(np.stack(mixed), width)
        np.testing.assert_array_equal(t_out[b].cpu().numpy(), wt)
        np.testing.assert_array_equal(i_out[b].cpu().numpy(), wi)
        np.testing.assert_array_equal(s_out[b].cpu().numpy(), wst)
        counts["trees"] += 1
        counts["trees_all_clear"] += int(all_clear)
    return counts
