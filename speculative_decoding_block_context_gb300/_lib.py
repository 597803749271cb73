"""Thin ctypes binding of libflashmap.so (include/flashmap.h).

Functions carry the C names and only marshal arguments: torch tensors become device
pointers, None becomes NULL, the current torch stream is passed when none is given.
Every step of the computation runs in the library's CUDA kernels; nothing here
computes. A missing library raises instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libflashmap.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "flashmap.h")

F32, BF16, E4M3 = 0, 1, 2
DTYPE_CODES = {"f32": F32, "bf16": BF16, "e4m3": E4M3}
STATUS = {0: "OK", 1: "E_INVALID", 2: "E_UNSUPPORTED", 3: "E_CUDA", 4: "E_NOMEM", 5: "E_DEVICE"}
DEVERR = {"PAGE": 1, "POSITION": 2, "TOKEN": 4, "TIMEOUT": 8, "NUMERIC": 16}

_c = ctypes
_vp = _c.c_void_p


class flashmap_config(_c.Structure):
    _fields_ = [(n, _c.c_int32) for n in (
        "target_hidden", "num_target_layers", "hidden", "num_layers", "num_heads", "head_dim",
        "intermediate", "cond_dim", "time_embed_dim", "block_size", "vocab_size", "draft_vocab_size",
        "num_steps", "noise_gate_constant", "page_size", "max_position")] + \
        [(n, _c.c_float) for n in ("time_scale", "rope_theta", "rms_norm_eps", "qk_norm_eps", "layer_norm_eps")] + \
        [("act_dtype", _c.c_int32), ("weight_dtype", _c.c_int32), ("kv_dtype", _c.c_int32),
         ("noise_path", _c.c_int32)]


LAYER_FIELDS = {
    "self_adaln_w": "self_attn_adaln.linear.weight", "self_adaln_b": "self_attn_adaln.linear.bias",
    "self_q_w": "self_attn.q_proj.weight", "self_k_w": "self_attn.k_proj.weight",
    "self_v_w": "self_attn.v_proj.weight", "self_o_w": "self_attn.o_proj.weight",
    "self_q_norm_w": "self_attn.q_norm.weight", "self_k_norm_w": "self_attn.k_norm.weight",
    "cross_adaln_w": "cross_attn_adaln.linear.weight", "cross_adaln_b": "cross_attn_adaln.linear.bias",
    "cross_q_w": "cross_attn.q_proj.weight", "cross_k_w": "cross_attn.k_proj.weight",
    "cross_v_w": "cross_attn.v_proj.weight", "cross_o_w": "cross_attn.o_proj.weight",
    "cross_q_norm_w": "cross_attn.q_norm.weight", "cross_k_norm_w": "cross_attn.k_norm.weight",
    "mlp_adaln_w": "mlp_adaln.linear.weight", "mlp_adaln_b": "mlp_adaln.linear.bias",
    "fc1_w": "mlp.fc1.weight", "fc1_b": "mlp.fc1.bias", "fc2_w": "mlp.fc2.weight", "fc2_b": "mlp.fc2.bias",
}
MODEL_FIELDS = {
    "fc_w": "fc.weight", "hidden_norm_w": "hidden_norm.weight", "anchor_proj_w": "anchor_proj.weight",
    "anchor_proj_b": "anchor_proj.bias", "anchor_norm_w": "anchor_norm.weight",
    "state_norm_w": "state_norm.weight", "noise_norm_w": "noise_norm.weight", "noise_gate": "noise_gate",
    "x_embed_w": "x_embed.weight", "x_embed_b": "x_embed.bias",
    "time_l1_w": "time_embed.linear_1.weight", "time_l1_b": "time_embed.linear_1.bias",
    "time_l2_w": "time_embed.linear_2.weight", "time_l2_b": "time_embed.linear_2.bias",
    "jump_l1_w": "jump_embed.linear_1.weight", "jump_l1_b": "jump_embed.linear_1.bias",
    "jump_l2_w": "jump_embed.linear_2.weight", "jump_l2_b": "jump_embed.linear_2.bias",
    "final_adaln_w": "final_adaln.linear.weight", "final_adaln_b": "final_adaln.linear.bias",
    "head_w": "head.weight", "head_b": "head.bias",
}


class flashmap_layer_weights(_c.Structure):
    _fields_ = [(n, _vp) for n in LAYER_FIELDS]


class flashmap_weights(_c.Structure):
    _fields_ = [(n, _vp) for n in MODEL_FIELDS] + [("layers", _c.POINTER(flashmap_layer_weights))]


class flashmap_kv_pool(_c.Structure):
    _fields_ = [("base", _vp), ("num_pages", _c.c_int64), ("dtype", _c.c_int32)]


class flashmap_pending_write(_c.Structure):
    _fields_ = [("target_hidden", _vp), ("W", _c.c_int32), ("start_pos", _vp), ("commit_lens", _vp),
                ("out_loc", _vp)]


class flashmap_launch_record(_c.Structure):
    _fields_ = [("kind", _c.c_int32), ("layer", _c.c_int32), ("rows", _c.c_int32), ("n", _c.c_int32),
                ("k", _c.c_int32), ("ms", _c.c_float)]


KINDS = {0: "gemm", 1: "xattn", 2: "xcombine", 3: "self_attn", 4: "rows", 5: "sample", 6: "memset"}


class FlashmapError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def lib():
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = _c.CDLL(LIB_PATH)
        st = _c.c_int
        P = _c.POINTER
        L.flashmap_last_error.restype = _c.c_char_p
        L.flashmap_validate_config.argtypes = [P(flashmap_config)]
        L.flashmap_pool_bytes.argtypes = [P(flashmap_config), _c.c_int64, P(_c.c_size_t)]
        L.flashmap_load_weights.argtypes = [P(flashmap_config), P(flashmap_weights), _vp, _vp, _vp, _vp, P(_vp)]
        L.flashmap_free.argtypes = [_vp]
        L.flashmap_get_config.argtypes = [_vp, P(flashmap_config)]
        L.flashmap_workspace_size.argtypes = [_vp, _c.c_int32, _c.c_int32, P(_c.c_size_t)]
        L.flashmap_write_context_kv.argtypes = [_vp, P(flashmap_kv_pool), _vp, _c.c_int32, _c.c_int32, _vp, _vp,
                                                _vp, _vp, _c.c_int32, _vp, _vp, _c.c_size_t, _vp]
        L.flashmap_draft_block.argtypes = [_vp, P(flashmap_kv_pool), _c.c_int32, _vp, _vp, _vp, _vp, _c.c_int32,
                                           _vp, _c.c_float, _vp, _vp, _vp, _c.c_size_t, _vp]
        L.flashmap_draft_block_with_write.argtypes = [_vp, P(flashmap_kv_pool), P(flashmap_pending_write), _c.c_int32,
                                                      _vp, _vp, _vp, _vp, _c.c_int32, _vp, _c.c_float, _vp, _vp, _vp,
                                                      _c.c_size_t, _vp]
        L.flashmap_sample_block.argtypes = [_vp, _c.c_int32, _vp, _vp, _vp, _vp, _vp, _c.c_uint64, _vp, _vp, _vp,
                                            _vp, _c.c_size_t, _vp]
        L.flashmap_get_device_error.argtypes = [_vp, _vp, P(_c.c_uint32)]
        L.flashmap_debug_philox.argtypes = [_vp, _vp, _c.c_int64, _vp, _vp, _vp]
        L.flashmap_debug_linear.argtypes = [_c.c_int32, _vp, _vp, _c.c_int32, _c.c_int32, _c.c_int32, _vp, _vp]
        L.flashmap_debug_constants.argtypes = [_vp, _vp, _vp, _vp, _vp]
        L.flashmap_debug_folded.argtypes = [_vp, _vp, _vp, _vp, P(_c.c_int32), _vp]
        L.flashmap_sample_logits_static.argtypes = [_vp, _c.c_int32, _vp, _vp, _vp, _vp, _vp, _c.c_uint64, _vp, _vp]
        L.flashmap_debug_wait_timeout.argtypes = [_vp, _c.c_uint64, _vp]
        L.flashmap_profile_gemm_chain.argtypes = [_vp, _c.c_int32, _c.c_int32, _vp, _vp, _c.c_size_t,
                                                  P(_c.c_int64), P(_c.c_int32), _vp]
        L.flashmap_build_tree.argtypes = [_vp, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32, _vp, _vp, _vp, _vp]
        L.flashmap_draft_candidates.argtypes = [_vp, P(flashmap_kv_pool), _c.c_int32, _c.c_int32, _vp, _vp, _vp, _vp,
                                                _c.c_int32, _vp, _c.c_float, _vp, _vp, _vp, _c.c_size_t, _vp]
        L.flashmap_profile_start.argtypes = [_vp, _c.c_int32]
        L.flashmap_profile_stop.argtypes = [_vp, P(flashmap_launch_record), _c.c_int32, P(_c.c_int32)]
        for name in header_functions():
            getattr(L, name).restype = st if name != "flashmap_last_error" else _c.c_char_p
        _lib = L
    return _lib


def header_functions() -> list:
    """Every function declared in include/flashmap.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:flashmap_status|const char\*)\s+(flashmap_\w+)\s*\(", text, re.M)))


def _check(status: int) -> None:
    if status != 0:
        raise FlashmapError(status, lib().flashmap_last_error().decode())


def _ptr(t):
    return None if t is None else _vp(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return _vp(stream)
    import torch

    return _vp(torch.cuda.current_stream().cuda_stream)


def make_config(d: dict) -> flashmap_config:
    c = flashmap_config()
    for name, ctype in flashmap_config._fields_:
        if name in ("act_dtype", "weight_dtype", "kv_dtype"):
            v = d.get(name, d["act_dtype"])  # the pool defaults to the activation dtype
            setattr(c, name, DTYPE_CODES[v] if isinstance(v, str) else int(v))
        elif ctype is _c.c_float:
            setattr(c, name, float(d[name]))
        else:
            setattr(c, name, int(d.get(name, 0)))
    return c


def flashmap_validate_config(cfg: dict) -> int:
    """Status of the config check (0 = OK); does not raise."""
    return lib().flashmap_validate_config(_c.byref(make_config(cfg)))


def flashmap_last_error() -> str:
    return lib().flashmap_last_error().decode()


def flashmap_pool_bytes(cfg: dict, num_pages: int) -> int:
    n = _c.c_size_t()
    _check(lib().flashmap_pool_bytes(_c.byref(make_config(cfg)), int(num_pages), _c.byref(n)))
    return n.value


class Model:
    """A loaded drafter handle plus the host structs that must outlive the load call."""

    def __init__(self, handle, cfg: dict, embedding):
        self.handle = handle
        self.cfg = cfg
        self._keep = embedding  # the library borrows the embedding

    def __del__(self):
        try:
            if self.handle:
                lib().flashmap_free(self.handle)
        except Exception:
            pass


def flashmap_load_weights(cfg: dict, weights: dict, embedding, lm_head, vocab_ranking=None, stream=None) -> Model:
    for t in list(weights.values()) + [embedding, lm_head]:
        if not t.is_contiguous():
            raise ValueError("weights must be contiguous device tensors")
    ccfg = make_config(cfg)
    layers = (flashmap_layer_weights * cfg["num_layers"])()
    for l in range(cfg["num_layers"]):
        for f, name in LAYER_FIELDS.items():
            setattr(layers[l], f, weights[f"layers.{l}.{name}"].data_ptr())
    w = flashmap_weights()
    for f, name in MODEL_FIELDS.items():
        setattr(w, f, weights[name].data_ptr())
    w.layers = layers
    out = _vp()
    _check(lib().flashmap_load_weights(_c.byref(ccfg), _c.byref(w), _ptr(embedding), _ptr(lm_head),
                                       _ptr(vocab_ranking), _stream(stream), _c.byref(out)))
    return Model(out, cfg, embedding)


def flashmap_workspace_size(model: Model, max_bs: int, max_write_rows: int) -> int:
    n = _c.c_size_t()
    _check(lib().flashmap_workspace_size(model.handle, int(max_bs), int(max_write_rows), _c.byref(n)))
    return n.value


def make_pool(pool_tensor, num_pages: int, dtype: int) -> flashmap_kv_pool:
    return flashmap_kv_pool(pool_tensor.data_ptr(), int(num_pages), int(dtype))


def flashmap_write_context_kv(model: Model, pool: flashmap_kv_pool, target_hidden, bs: int, W: int, req_pool_idx,
                              start_pos, commit_lens, req_to_page, out_loc, workspace, stream=None) -> None:
    _check(lib().flashmap_write_context_kv(
        model.handle, _c.byref(pool), _ptr(target_hidden), int(bs), int(W), _ptr(req_pool_idx), _ptr(start_pos),
        _ptr(commit_lens), _ptr(req_to_page), int(req_to_page.stride(0)), _ptr(out_loc), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def flashmap_draft_block(model: Model, pool: flashmap_kv_pool, bs: int, anchor_ids, anchor_pos, req_pool_idx,
                         req_to_page, seeds, noise_scale: float, hidden_out, anchor_loc_out, workspace,
                         stream=None) -> None:
    _check(lib().flashmap_draft_block(
        model.handle, _c.byref(pool), int(bs), _ptr(anchor_ids), _ptr(anchor_pos), _ptr(req_pool_idx),
        _ptr(req_to_page), int(req_to_page.stride(0)), _ptr(seeds), float(noise_scale), _ptr(hidden_out),
        _ptr(anchor_loc_out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def flashmap_draft_block_with_write(model: Model, pool: flashmap_kv_pool, target_hidden, W: int, start_pos, commit_lens,
                                    out_loc, bs: int, anchor_ids, anchor_pos, req_pool_idx, req_to_page, seeds,
                                    noise_scale: float, hidden_out, anchor_loc_out, workspace, stream=None) -> None:
    pending = flashmap_pending_write(_ptr(target_hidden), int(W), _ptr(start_pos), _ptr(commit_lens), _ptr(out_loc))
    _check(lib().flashmap_draft_block_with_write(
        model.handle, _c.byref(pool), _c.byref(pending), int(bs), _ptr(anchor_ids), _ptr(anchor_pos),
        _ptr(req_pool_idx), _ptr(req_to_page), int(req_to_page.stride(0)), _ptr(seeds), float(noise_scale),
        _ptr(hidden_out), _ptr(anchor_loc_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def flashmap_draft_candidates(model: Model, pool: flashmap_kv_pool, bs: int, n_cand: int, anchor_ids, anchor_pos,
                              req_pool_idx, req_to_page, seeds, noise_scale: float, hidden_out, anchor_loc_out,
                              workspace, stream=None) -> None:
    _check(lib().flashmap_draft_candidates(
        model.handle, _c.byref(pool), int(bs), int(n_cand), _ptr(anchor_ids), _ptr(anchor_pos), _ptr(req_pool_idx),
        _ptr(req_to_page), int(req_to_page.stride(0)), _ptr(seeds), float(noise_scale), _ptr(hidden_out),
        _ptr(anchor_loc_out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def flashmap_sample_block(model: Model, bs: int, hidden, anchor_pos, temperature, greedy, seeds, step: int,
                          tokens_out, draft_logits_out, full_logits_out, workspace, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().flashmap_sample_block(
        model.handle, int(bs), _ptr(hidden), _ptr(anchor_pos), _ptr(temperature), _ptr(greedy), _ptr(seeds),
        int(step), _ptr(tokens_out), _ptr(draft_logits_out), _ptr(full_logits_out), _ptr(workspace), ws_bytes,
        _stream(stream)))


def flashmap_sample_logits_static(model: Model, bs: int, logits, anchor_pos, temperature, greedy, seeds, step: int,
                                  tokens_out, stream=None) -> None:
    """Sampling from caller-provided logits with the library's static scratch (no
    device allocation; at most 8192 rows; overlapping calls race)."""
    _check(lib().flashmap_sample_logits_static(model.handle, int(bs), _ptr(logits), _ptr(anchor_pos),
                                               _ptr(temperature), _ptr(greedy), _ptr(seeds), int(step),
                                               _ptr(tokens_out), _stream(stream)))


def flashmap_build_tree(candidates, width: int, tokens_out, ids_out, stats_out, stream=None) -> None:
    """candidates (bs, n_cand, block_size) int64 device -> the verify tree (in place)."""
    bs, n, k = candidates.shape
    _check(lib().flashmap_build_tree(_ptr(candidates), int(bs), int(n), int(k), int(width), _ptr(tokens_out),
                                     _ptr(ids_out), _ptr(stats_out), _stream(stream)))


def flashmap_get_device_error(model: Model, stream=None) -> int:
    code = _c.c_uint32()
    st = lib().flashmap_get_device_error(model.handle, _stream(stream), _c.byref(code))
    if st not in (0, 5):
        _check(st)
    return code.value


def flashmap_debug_philox(seeds, ctr, out, normals=None, stream=None) -> None:
    _check(lib().flashmap_debug_philox(_ptr(seeds), _ptr(ctr), int(seeds.numel()), _ptr(out), _ptr(normals),
                                       _stream(stream)))


def flashmap_debug_linear(dtype: int, x, w, out, stream=None) -> None:
    rows, k = x.shape
    n = w.shape[0]
    _check(lib().flashmap_debug_linear(int(dtype), _ptr(x), _ptr(w), int(rows), int(k), int(n), _ptr(out),
                                       _stream(stream)))


def flashmap_debug_constants(model: Model, chol=None, uniform=None, hot_ids=None, stream=None) -> None:
    _check(lib().flashmap_debug_constants(model.handle, _ptr(chol), _ptr(uniform), _ptr(hot_ids), _stream(stream)))


def flashmap_debug_folded(model: Model, variance=None, embedded_uniform=None, proj=None, stream=None) -> int:
    """Copies the folded-noise constants; returns the Jacobi sweeps the load took."""
    sweeps = _c.c_int32(0)
    _check(lib().flashmap_debug_folded(model.handle, _ptr(variance), _ptr(embedded_uniform), _ptr(proj),
                                       _c.byref(sweeps), _stream(stream)))
    return int(sweeps.value)


def flashmap_profile_start(model: Model, capacity: int = 4096) -> None:
    _check(lib().flashmap_profile_start(model.handle, int(capacity)))


def flashmap_profile_stop(model: Model, capacity: int = 4096) -> list:
    """Launch records [(kind name, layer, rows, n, k, ms)] since flashmap_profile_start."""
    recs = (flashmap_launch_record * capacity)()
    n = _c.c_int32()
    _check(lib().flashmap_profile_stop(model.handle, recs, int(capacity), _c.byref(n)))
    return [(KINDS.get(r.kind, str(r.kind)), r.layer, r.rows, r.n, r.k, r.ms) for r in recs[: min(n.value, capacity)]]


def flashmap_profile_gemm_chain(model: Model, bs: int, window: int, hidden, workspace, stream=None) -> tuple:
    """Launches the GEMMs of one step back to back (see the header); returns
    (algorithmic bytes, launches)."""
    b = _c.c_int64()
    n = _c.c_int32()
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().flashmap_profile_gemm_chain(model.handle, int(bs), int(window), _ptr(hidden), _ptr(workspace),
                                             ws_bytes, _c.byref(b), _c.byref(n), _stream(stream)))
    return b.value, n.value


def flashmap_debug_wait_timeout(model: Model, limit_ns: int, stream=None) -> None:
    """One warp waits limit_ns on an mbarrier nothing arrives on and reports the timeout."""
    _check(lib().flashmap_debug_wait_timeout(model.handle, int(limit_ns), _stream(stream)))
