"""PyTorch-facing binding of libmla: argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module checks
tensor placement/dtypes, allocates outputs and the workspace with torch when the
caller does not pass them, and forwards raw pointers and the current stream.
There is no CPU fallback: without a CUDA device or the built library every call
raises.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import numpy as np
import torch

from . import _lib
from ._lib import (KV_BF16, KV_FP8_E4M3, OUT_BF16, OUT_FP32, PART_ALL, PART_CONTEXT,  # noqa: F401
                   PART_EXTEND, MLAError)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return ctypes.c_void_p(t.data_ptr())


def set_kernel_events(begin: Optional[torch.cuda.Event], end: Optional[torch.cuda.Event]) -> None:
    """Time the fused prefill kernel of later prefill() calls with these events
    (recorded on the call's stream around the fused kernel launches)."""
    if begin is None or end is None:
        _lib.load().mla_set_kernel_events(None, None)
        return
    for e in (begin, end):      # torch creates the CUDA event lazily on first record
        if not e.cuda_event:
            e.record()
    _lib.load().mla_set_kernel_events(ctypes.c_void_p(begin.cuda_event), ctypes.c_void_p(end.cuda_event))


def launch_count() -> int:
    """Kernels launched by libmla so far in this process."""
    return int(_lib.load().mla_launch_count())


def kv_dtype_code(kv_cache: torch.Tensor) -> int:
    if kv_cache.dtype == torch.bfloat16 and kv_cache.shape[-1] == 576:
        return KV_BF16
    if kv_cache.dtype == torch.uint8 and kv_cache.shape[-1] == 640:
        return KV_FP8_E4M3
    raise ValueError("kv_cache must be bf16 [NB,64,576] or uint8 [NB,64,640]")


def prefill_workspace_size(seq_lens, cu_q, num_heads: int, segments=None, chunk: int = 4096,
                           parts: int = PART_ALL) -> int:
    sl, _k1 = _lib.i32_host(seq_lens)
    cq, _k2 = _lib.i32_host(cu_q)
    sp, ns, _k3 = _lib.segments_host(segments)
    n = _lib.load().mla_prefill_workspace_size(len(_k1), sl, cq, int(num_heads), sp, ns, int(chunk), int(parts))
    if n == 0:
        raise MLAError("mla_prefill_workspace_size", _lib.MLA_ERR_INVALID_ARG)
    return int(n)


def prefill_min_workspace_size(seq_lens, cu_q, num_heads: int, segments=None, chunk: int = 4096,
                               parts: int = PART_ALL) -> int:
    """The smallest workspace mla_prefill_ctx runs in (shallow K/V rings, one
    piece per launch: slower)."""
    sl, _k1 = _lib.i32_host(seq_lens)
    cq, _k2 = _lib.i32_host(cu_q)
    sp, ns, _k3 = _lib.segments_host(segments)
    n = _lib.load().mla_prefill_min_workspace_size(len(_k1), sl, cq, int(num_heads), sp, ns, int(chunk), int(parts))
    if n == 0:
        raise MLAError("mla_prefill_min_workspace_size", _lib.MLA_ERR_INVALID_ARG)
    return int(n)


def absorbed_workspace_size(seq_lens, cu_q, num_heads: int, segments=None, chunk: int = 4096,
                            parts: int = PART_ALL, fp8_scores: bool = False) -> int:
    sl, _k1 = _lib.i32_host(seq_lens)
    cq, _k2 = _lib.i32_host(cu_q)
    sp, ns, _k3 = _lib.segments_host(segments)
    L = _lib.load()
    fn = L.mla_prefill_absorbed_fp8_workspace_size if fp8_scores else L.mla_prefill_absorbed_workspace_size
    if fp8_scores == "auto":
        fn = L.mla_prefill_auto_workspace_size
    n = fn(len(_k1), sl, cq, int(num_heads), sp, ns, int(chunk), int(parts))
    if n == 0:
        raise MLAError("mla_prefill_absorbed_workspace_size", _lib.MLA_ERR_INVALID_ARG)
    return int(n)


def prefill(q: torch.Tensor, q_pos: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
            seq_lens, cu_q, kv_b_proj: torch.Tensor, *, chunk: int, softmax_scale: float,
            rope_theta: float = 10000.0, kv_scale: float = 1.0, segments=None, parts: int = PART_ALL,
            out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
            lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None, absorbed=False,
            kv_b_proj_e4m3: Optional[torch.Tensor] = None, w_scale: Optional[float] = None
            ) -> Tuple[torch.Tensor, torch.Tensor]:
    """MLA chunked prefill of one layer (mla_prefill_ctx; absorbed=True:
    mla_prefill_ctx_absorbed, the same result computed in latent space;
    absorbed="fp8": mla_prefill_ctx_absorbed_fp8, FP8 caches, latent scores
    on the FP8 tensor cores; absorbed="auto": mla_prefill_ctx_auto, the path
    chosen per request by its number of queries).  With kv_b_proj_e4m3 (uint8
    [H*256, 512], see kv_b_proj_to_e4m3) and w_scale: mla_prefill_ctx_fp8w,
    FP8 caches, the up-projection on the FP8 tensor cores.

    q bf16 [T_q, H, 192] (q_rope unrotated); q_pos int32 [T_q]; kv_cache bf16
    [NB,64,576] or uint8 [NB,64,640] (FP8); block_table int32 [B, max_blocks];
    seq_lens / cu_q host int32 (numpy or lists); kv_b_proj bf16 [512, H*256];
    segments optional host [S,4] (req, start, len, rope_offset).
    Returns (out [T_q, H, 128] in out_dtype, lse fp32 [T_q, H])."""
    T_q, H = int(q.shape[0]), int(q.shape[1])
    L = _lib.load()
    sl, keep_sl = _lib.i32_host(seq_lens)
    cq, keep_cq = _lib.i32_host(cu_q)
    sp, ns, keep_sp = _lib.segments_host(segments)
    B = int(keep_sl.shape[0])
    if keep_cq.shape[0] != B + 1 or int(keep_cq[-1]) != T_q:
        raise ValueError("cu_q must have num_reqs+1 entries ending at T_q")
    dev = q.device
    if out is None:
        out = torch.empty((T_q, H, 128), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T_q, H), dtype=torch.float32, device=dev)
    fp8 = absorbed == "fp8"
    auto = absorbed == "auto"
    fp8w = kv_b_proj_e4m3 is not None
    if fp8w and (absorbed or w_scale is None):
        raise ValueError("kv_b_proj_e4m3 takes w_scale and the up-projected path")
    if workspace is None:
        if absorbed:
            ws_bytes = absorbed_workspace_size(keep_sl, keep_cq, H, segments, chunk, parts,
                                               fp8_scores="auto" if auto else fp8)
        else:
            ws_bytes = prefill_workspace_size(keep_sl, keep_cq, H, segments, chunk, parts)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    od = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_FP32
    common = (_dev(q, "q", torch.bfloat16), _dev(q_pos, "q_pos", torch.int32), _dev(kv_cache, "kv_cache"),
              kv_dtype_code(kv_cache), float(kv_scale), int(kv_cache.shape[0]),
              _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
              sl, cq, B, H, sp, ns, int(chunk))
    tail = (float(softmax_scale), float(rope_theta), int(parts),
            _dev(out, "out", (torch.float32, torch.bfloat16)), od, _dev(lse, "lse", torch.float32),
            _dev(workspace, "workspace"), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
            _stream_ptr(stream))
    if fp8w:
        name = "mla_prefill_ctx_fp8w"
        st = L.mla_prefill_ctx_fp8w(*common, _dev(kv_b_proj_e4m3, "kv_b_proj_e4m3", torch.uint8), float(w_scale),
                                    *tail)
    else:
        name = ("mla_prefill_ctx_auto" if auto else "mla_prefill_ctx_absorbed_fp8" if fp8
                else "mla_prefill_ctx_absorbed" if absorbed else "mla_prefill_ctx")
        st = getattr(L, name)(*common, _dev(kv_b_proj, "kv_b_proj", torch.bfloat16), *tail)
    _lib.check(name, st)
    prefill.last_workspace = workspace
    return out, lse


def kv_b_proj_absmax(kv_b_proj: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> float:
    """The largest |w| of a bf16 kv_b_proj [512, H*256] (mla_kv_b_proj_absmax; synchronises)."""
    H = int(kv_b_proj.shape[1]) // 256
    out = torch.empty(1, dtype=torch.float32, device=kv_b_proj.device)
    _lib.check("mla_kv_b_proj_absmax", _lib.load().mla_kv_b_proj_absmax(
        _dev(kv_b_proj, "kv_b_proj", torch.bfloat16), H, _dev(out, "absmax"), _stream_ptr(stream)))
    return float(out.item())


def kv_b_proj_to_e4m3(kv_b_proj: torch.Tensor, w_scale: float, out: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """E4M3 codes of kv_b_proj / w_scale, transposed: uint8 [H*256, 512]
    (mla_kv_b_proj_to_e4m3).  w_scale = absmax / 448 uses the whole range."""
    cols = int(kv_b_proj.shape[1])
    if out is None:
        out = torch.empty((cols, 512), dtype=torch.uint8, device=kv_b_proj.device)
    _lib.check("mla_kv_b_proj_to_e4m3", _lib.load().mla_kv_b_proj_to_e4m3(
        _dev(kv_b_proj, "kv_b_proj", torch.bfloat16), cols // 256, float(w_scale), _dev(out, "out", torch.uint8),
        _stream_ptr(stream)))
    return out


def _protected_host(protected_rows, T_q: int):
    if protected_rows is None:
        return None, None
    m = np.zeros(T_q, dtype=np.uint8)
    pr = np.asarray(protected_rows)
    if pr.dtype == bool and pr.shape == (T_q,):
        m[:] = pr
    else:
        m[pr.astype(np.int64)] = 1
    return ctypes.c_void_p(m.ctypes.data), m


def reuse_workspace_size(seq_lens, cu_q, num_heads: int, global_heads, protected_rows=None, segments=None,
                         chunk: int = 4096, parts: int = PART_ALL) -> int:
    sl, keep_sl = _lib.i32_host(seq_lens)
    cq, keep_cq = _lib.i32_host(cu_q)
    sp, ns, _k3 = _lib.segments_host(segments)
    gh, keep_gh = _lib.i32_host(list(global_heads))
    pp, _k4 = _protected_host(protected_rows, int(keep_cq[-1]))
    n = _lib.load().mla_prefill_reuse_workspace_size(len(keep_sl), sl, cq, int(num_heads), sp, ns, int(chunk),
                                                     int(parts), gh, int(keep_gh.shape[0]), pp)
    if n == 0:
        raise MLAError("mla_prefill_reuse_workspace_size", _lib.MLA_ERR_INVALID_ARG)
    return int(n)


def prefill_reuse(q: torch.Tensor, q_pos: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                  seq_lens, cu_q, kv_b_proj: torch.Tensor, art_out: torch.Tensor, art_lse: torch.Tensor, *,
                  global_heads, protected_rows=None, chunk: int, softmax_scale: float, rope_theta: float = 10000.0,
                  kv_scale: float = 1.0, segments=None, parts: int = PART_ALL,
                  out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
                  lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Head-split reuse (mla_prefill_reuse): the Global heads and the
    protected rows (host indices or a bool mask over T_q) are recomputed,
    every other (row, head) takes the artifact (art_out fp32 [T_q, H, 128],
    art_lse fp32 [T_q, H])."""
    T_q, H = int(q.shape[0]), int(q.shape[1])
    sl, keep_sl = _lib.i32_host(seq_lens)
    cq, keep_cq = _lib.i32_host(cu_q)
    sp, ns, keep_sp = _lib.segments_host(segments)
    gh, keep_gh = _lib.i32_host(list(global_heads))
    pp, keep_pp = _protected_host(protected_rows, T_q)
    dev = q.device
    if out is None:
        out = torch.empty((T_q, H, 128), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T_q, H), dtype=torch.float32, device=dev)
    if workspace is None:
        ws_bytes = reuse_workspace_size(keep_sl, keep_cq, H, keep_gh, keep_pp.astype(bool) if keep_pp is not None
                                        else None, segments, chunk, parts)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    od = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_FP32
    st = _lib.load().mla_prefill_reuse(
        _dev(q, "q", torch.bfloat16), _dev(q_pos, "q_pos", torch.int32), _dev(kv_cache, "kv_cache"),
        kv_dtype_code(kv_cache), float(kv_scale), int(kv_cache.shape[0]),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        sl, cq, int(keep_sl.shape[0]), H, sp, ns, int(chunk), _dev(kv_b_proj, "kv_b_proj", torch.bfloat16),
        float(softmax_scale), float(rope_theta), int(parts), gh, int(keep_gh.shape[0]), pp,
        _dev(art_out, "art_out", torch.float32), _dev(art_lse, "art_lse", torch.float32),
        _dev(out, "out", (torch.float32, torch.bfloat16)), od, _dev(lse, "lse", torch.float32),
        _dev(workspace, "workspace"), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
        _stream_ptr(stream))
    _lib.check("mla_prefill_reuse", st)
    prefill_reuse.last_workspace = workspace
    return out, lse


def device_error(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Reads and clears the device error word of a prefill workspace."""
    return int(_lib.load().mla_get_device_error(_dev(workspace, "workspace"), _stream_ptr(stream)))


def merge_states(out_a, lse_a, out_b, lse_b, out=None, lse=None, stream=None):
    """merge_attn_states on fp32 [rows, d_v] states and fp32 [rows] lse."""
    d_v = int(out_a.shape[-1])
    rows = int(out_a.numel() // d_v)
    out = torch.empty_like(out_a) if out is None else out
    lse = torch.empty_like(lse_a) if lse is None else lse
    f32 = torch.float32
    st = _lib.load().mla_merge_states(_dev(out_a, "out_a", f32), _dev(lse_a, "lse_a", f32), _dev(out_b, "out_b", f32),
                                      _dev(lse_b, "lse_b", f32), _dev(out, "out", f32), _dev(lse, "lse", f32),
                                      rows, d_v, _stream_ptr(stream))
    _lib.check("mla_merge_states", st)
    return out, lse


def rope_relocate(x: torch.Tensor, pos: torch.Tensor, offset: int, theta: float = 10000.0,
                  y: Optional[torch.Tensor] = None, rope_col: Optional[int] = None, stream=None) -> torch.Tensor:
    """Rotate the 64 RoPE columns of bf16 x [tokens, heads, row] by (pos - offset)."""
    tokens, heads, row = int(x.shape[0]), int(x.shape[1]), int(x.shape[2])
    rope_col = row - 64 if rope_col is None else int(rope_col)
    if y is None:
        y = x.clone()
    st = _lib.load().mla_rope_relocate(_dev(x, "x", torch.bfloat16), _dev(pos, "pos", torch.int32), int(offset),
                                       float(theta), _dev(y, "y", torch.bfloat16), tokens, heads, row, rope_col,
                                       _stream_ptr(stream))
    _lib.check("mla_rope_relocate", st)
    return y


def gather_latent(kv_cache: torch.Tensor, block_table_row: torch.Tensor, start: int, length: int,
                  kv_scale: float = 1.0, dst: Optional[torch.Tensor] = None,
                  dev_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Rows of tokens [start, start+length) of one request as bf16 [length, 576]."""
    if dst is None:
        dst = torch.empty((length, 576), dtype=torch.bfloat16, device=kv_cache.device)
    errp = _dev(dev_error, "dev_error", (torch.int32, torch.uint32)) if dev_error is not None else None
    st = _lib.load().mla_gather_latent(_dev(kv_cache, "kv_cache"), kv_dtype_code(kv_cache), float(kv_scale),
                                       int(kv_cache.shape[0]), _dev(block_table_row, "block_table_row", torch.int32),
                                       int(block_table_row.shape[0]), int(start), int(length),
                                       _dev(dst, "dst", torch.bfloat16), errp, _stream_ptr(stream))
    _lib.check("mla_gather_latent", st)
    return dst


def block_hash(kv_cache: torch.Tensor, block_ids: torch.Tensor, dev_error: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """Content hash of whole cache blocks (mla_block_hash): int64 [n] holding
    the uint64 hash bits."""
    n = int(block_ids.numel())
    hashes = torch.empty(n, dtype=torch.int64, device=kv_cache.device)
    errp = _dev(dev_error, "dev_error", (torch.int32, torch.uint32)) if dev_error is not None else None
    st = _lib.load().mla_block_hash(_dev(kv_cache, "kv_cache"), kv_dtype_code(kv_cache), int(kv_cache.shape[0]),
                                    _dev(block_ids, "block_ids", torch.int32), n, _dev(hashes, "hashes"), errp,
                                    _stream_ptr(stream))
    _lib.check("mla_block_hash", st)
    return hashes


def block_compare(kv_cache: torch.Tensor, block_a: torch.Tensor, block_b: torch.Tensor,
                  dev_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Byte equality of block pairs (mla_block_compare): int32 [n], 1 equal, 0 not."""
    n = int(block_a.numel())
    if int(block_b.numel()) != n:
        raise ValueError("block_a and block_b differ in length")
    equal = torch.empty(n, dtype=torch.int32, device=kv_cache.device)
    errp = _dev(dev_error, "dev_error", (torch.int32, torch.uint32)) if dev_error is not None else None
    st = _lib.load().mla_block_compare(_dev(kv_cache, "kv_cache"), kv_dtype_code(kv_cache), int(kv_cache.shape[0]),
                                       _dev(block_a, "block_a", torch.int32), _dev(block_b, "block_b", torch.int32),
                                       n, _dev(equal, "equal"), errp, _stream_ptr(stream))
    _lib.check("mla_block_compare", st)
    return equal


# ---------------------------------------------------------------- workloads

class DeviceWorkload:
    """Device copies of a workload's inputs (see workload.Workload)."""

    def __init__(self, wl, device="cuda"):
        self.wl = wl
        dev = torch.device(device)
        self.q = torch.from_numpy(wl.q.view(np.int16)).to(dev).view(torch.bfloat16)
        self.q_pos = torch.from_numpy(wl.q_pos).to(dev)
        if wl.kv_dtype == "bf16":
            self.kv_cache = torch.from_numpy(wl.kv_cache.view(np.int16)).to(dev).view(torch.bfloat16)
        else:
            self.kv_cache = torch.from_numpy(wl.kv_cache).to(dev)
        self.block_table = torch.from_numpy(wl.block_table).to(dev)
        self.kv_b_proj = torch.from_numpy(wl.kv_b_proj.view(np.int16)).to(dev).view(torch.bfloat16)
        self.seq_lens = wl.seq_lens
        self.cu_q = wl.cu_q

    def run(self, parts=PART_ALL, out_dtype=torch.float32, chunk=None, **kw):
        wl = self.wl
        return prefill(self.q, self.q_pos, self.kv_cache, self.block_table, self.seq_lens, self.cu_q,
                       self.kv_b_proj, chunk=wl.chunk if chunk is None else chunk,
                       softmax_scale=wl.softmax_scale, rope_theta=wl.rope_theta, kv_scale=wl.kv_scale,
                       segments=wl.segments, parts=parts, out_dtype=out_dtype, **kw)
