"""Python binding of libdcp_gb300 (sharded absorbed-MLA decode for GB300 / sm_103a).

Argument marshalling only: every function takes torch tensors that already live
on the GPU, checks their dtype/shape/contiguity, and forwards raw device
pointers plus the current CUDA stream to the C ABI declared in
``include/dcp.h``.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU path.  If the library has not been built, importing
works but the first call raises ``RuntimeError``.

Functions (same names as the C ABI):
  dcp_count, dcp_slot_map, dcp_kv_append, dcp_mla_decode_partial,
  dcp_mla_decode_workspace_size, dcp_lse_merge, dcp_kv_relayout, dcp_absorb_q,
  dcp_absorb_o, dcp_lse_merge_absorb_o, dcp_a2a_chunk_bytes, dcp_pack_partials,
  dcp_lse_merge_packed, dcp_lse_rescale
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "DcpError", "Layout", "load_library", "library_path",
    "dcp_count", "dcp_slot_map", "dcp_kv_append", "dcp_mla_decode_partial",
    "dcp_mla_decode_workspace_size", "dcp_lse_merge", "dcp_launch_count", "dcp_kv_relayout",
    "dcp_mla_decode_partial_static", "dcp_mla_decode_static_scratch_bytes", "dcp_absorb_q", "dcp_absorb_o",
    "dcp_a2a_chunk_bytes", "dcp_pack_partials", "dcp_lse_merge_packed", "dcp_lse_rescale", "dcp_lse_merge_absorb_o",
    "DCP_LSE_BASE_E", "DCP_LSE_BASE_2", "DCP_F32", "DCP_BF16", "STATUS_BITS",
]

DCP_OK, DCP_ERR_INVALID, DCP_ERR_UNSUPPORTED, DCP_ERR_CUDA, DCP_ERR_WORKSPACE = 0, -1, -2, -3, -4
DCP_ERR_TOO_LARGE = -5
DCP_LSE_BASE_E, DCP_LSE_BASE_2 = 0, 1
DCP_F32, DCP_BF16 = 0, 1
STATUS_BITS = {1: "BAD_POSITION", 2: "BAD_PAGE_INDEX", 4: "BAD_PAGE_ID", 8: "BAD_REQUEST", 16: "BAD_LENGTH",
               32: "TIMEOUT", 64: "INTERNAL"}


class DcpError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed with {code} ({msg})")
        self.code = code


class Layout(ctypes.Structure):
    """dcp_layout_t: n_shards N, interleave I (1 = token round-robin), page_size P."""
    _fields_ = [("n_shards", ctypes.c_int32), ("interleave", ctypes.c_int32), ("page_size", ctypes.c_int32)]

    def __repr__(self):
        return f"Layout(N={self.n_shards}, I={self.interleave}, P={self.page_size})"


_lib = None
_c = ctypes
_P = ctypes.c_void_p
_I32, _I64, _SZ, _F = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_LP = ctypes.POINTER(Layout)

_SIGNATURES = {
    "dcp_version": (_I32, []),
    "dcp_launch_count": (_I64, []),
    "dcp_error_string": (ctypes.c_char_p, [_I32]),
    "dcp_count": (_I64, [_LP, _I32, _I64]),
    "dcp_slot_map": (_I32, [_LP, _P, _P, _I64, _P, _I32, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "dcp_kv_append": (_I32, [_LP, _I32, _I32, _P, _P, _P, _I64, _P, _I32, _I64, _I64, _P, _I64, _P, _P]),
    "dcp_kv_relayout": (_I32, [_LP, _I32, _I32, _P, _I64, _I32, _P, _I64, _I64, _P, _P, _I64, _I32, _P, _I64, _I64,
                               _P, _I64, _P, _P]),
    "dcp_mla_decode_partial": (_I32, [_LP, _I32, _I32, _P, _I32, _I32, _I32, _P, _I64, _P, _I64, _I64,
                                      _P, _F, _I32, _P, _I32, _P, _P, _SZ, _P, _P]),
    "dcp_mla_decode_workspace_size": (_SZ, [_LP, _I32, _I32, _I32, _I32, _I32]),
    "dcp_lse_merge": (_I32, [_I32, _I64, _P, _I32, _P, _I32, _P, _I32, _P, _P]),
    "dcp_mla_decode_partial_static": (_I32, [_LP, _I32, _I32, _P, _I32, _I32, _I32, _P, _I64, _P, _I64, _I64,
                                             _P, _F, _I32, _P, _I32, _P, _P, _P]),
    "dcp_mla_decode_static_scratch_bytes": (_SZ, []),
    "dcp_absorb_q": (_I32, [_I64, _I32, _P, _I64, _P, _I64, _P, _P, _P, _P]),
    "dcp_absorb_o": (_I32, [_I64, _I32, _P, _I32, _P, _P, _I32, _P, _P]),
    "dcp_lse_merge_absorb_o": (_I32, [_I32, _I64, _I32, _P, _I32, _P, _I32, _P, _P, _I32, _P, _P, _P]),
    "dcp_a2a_chunk_bytes": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "dcp_pack_partials": (_I32, [_I32, _I32, _I32, _I32, _P, _I32, _P, _P, _I32, _P]),
    "dcp_lse_merge_packed": (_I32, [_I32, _I32, _I64, _P, _I32, _I32, _P, _I32, _P, _P]),
    "dcp_lse_rescale": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _I32, _I32, _P, _P, _P]),
}


def library_path() -> str:
    return _build.lib_path()


def load_library():
    """Load libdcp_gb300.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn, code):
    if code != DCP_OK:
        msg = load_library().dcp_error_string(code).decode()
        raise DcpError(fn, code, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return DCP_F32
    if t.dtype == torch.bfloat16:
        return DCP_BF16
    raise ValueError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def dcp_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load_library().dcp_launch_count())


def dcp_count(layout: Layout, shard: int, x: int) -> int:
    """Positions in [0, x) owned by `shard` (host-only)."""
    v = load_library().dcp_count(ctypes.byref(layout), shard, x)
    if v < 0:
        raise DcpError("dcp_count", DCP_ERR_INVALID, "invalid argument")
    return int(v)


def dcp_slot_map(layout, pos, req, block_table, max_pages, pool_pages, owner, row, slot, status, stream=None):
    """(owner, local row, slot) of each new token; writes into owner/row/slot."""
    T = pos.numel()
    _dev(pos, "pos", torch.int64, (T,))
    _dev(req, "req", torch.int32, (T,))
    _dev(block_table, "block_table", torch.int32)
    _dev(owner, "owner", torch.int32, (T,))
    _dev(row, "row", torch.int64, (T,))
    _dev(slot, "slot", torch.int64, (T,))
    _dev(status, "status", torch.int32, (1,))
    B, stride = block_table.shape
    _check("dcp_slot_map", load_library().dcp_slot_map(
        ctypes.byref(layout), _ptr(pos), _ptr(req), T, _ptr(block_table), B, stride, max_pages, pool_pages,
        _ptr(owner), _ptr(row), _ptr(slot), _ptr(status), _stream(stream)))


def dcp_kv_append(layout, shard_begin, shard_end, kv_new, pos, req, block_table, max_pages, arena, pool_pages,
                  status, stream=None):
    """Owner-filtered write of kv_new [T, 576] bf16 (positions pos, requests req) into
    arena [shards, pool_pages*P, 576]; placement computed in the same kernel."""
    T = kv_new.shape[0]
    _dev(kv_new, "kv_new", torch.bfloat16, (T, 576))
    _dev(pos, "pos", torch.int64, (T,))
    _dev(req, "req", torch.int32, (T,))
    _dev(block_table, "block_table", torch.int32)
    _dev(arena, "arena", torch.bfloat16, (shard_end - shard_begin, pool_pages * layout.page_size, 576))
    _dev(status, "status", torch.int32, (1,))
    B, stride = block_table.shape
    _check("dcp_kv_append", load_library().dcp_kv_append(
        ctypes.byref(layout), shard_begin, shard_end, _ptr(kv_new), _ptr(pos), _ptr(req), T, _ptr(block_table),
        B, stride, max_pages, _ptr(arena), pool_pages, _ptr(status), _stream(stream)))


def dcp_kv_relayout(layout, shard_begin, shard_end, src_pool, src_page_size, src_block_table, src_max_pages,
                    pos, req, block_table, max_pages, arena, pool_pages, status, stream=None):
    """Owner-filtered copy of tokens (pos, req) from a paged prefill pool src_pool [rows, 576] bf16."""
    T = pos.shape[0]
    _dev(src_pool, "src_pool", torch.bfloat16)
    if src_pool.dim() != 2 or src_pool.shape[1] != 576:
        raise ValueError("src_pool must be [rows, 576]")
    _dev(src_block_table, "src_block_table", torch.int32)
    _dev(pos, "pos", torch.int64, (T,))
    _dev(req, "req", torch.int32, (T,))
    _dev(block_table, "block_table", torch.int32)
    _dev(arena, "arena", torch.bfloat16, (shard_end - shard_begin, pool_pages * layout.page_size, 576))
    _dev(status, "status", torch.int32, (1,))
    B, stride = block_table.shape
    if src_block_table.shape[0] != B:
        raise ValueError("src_block_table and block_table must have one row per request")
    _check("dcp_kv_relayout", load_library().dcp_kv_relayout(
        ctypes.byref(layout), shard_begin, shard_end, _ptr(src_pool), src_pool.shape[0], src_page_size,
        _ptr(src_block_table), src_block_table.shape[1], src_max_pages, _ptr(pos), _ptr(req), T, B,
        _ptr(block_table), stride, max_pages, _ptr(arena), pool_pages, _ptr(status), _stream(stream)))


def dcp_mla_decode_workspace_size(layout, shard_begin, shard_end, B, q_len, H) -> int:
    return int(load_library().dcp_mla_decode_workspace_size(
        ctypes.byref(layout), shard_begin, shard_end, B, q_len, H))


def dcp_mla_decode_partial(layout, shard_begin, shard_end, q, arena, pool_pages, block_table, max_pages,
                           seq_lens, scale, lse_base, o_part, lse_part, workspace, status, stream=None):
    """Partials (o_r, lse_r) of shards [shard_begin, shard_end) for q [B, q_len, H, 576]."""
    B, q_len, H, dk = q.shape
    n = shard_end - shard_begin
    _dev(q, "q", torch.bfloat16, (B, q_len, H, 576))
    _dev(arena, "arena", torch.bfloat16, (n, pool_pages * layout.page_size, 576))
    _dev(block_table, "block_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int64, (B,))
    _dev(o_part, "o_part", o_part.dtype, (n, B, q_len, H, 512))
    _dev(lse_part, "lse_part", torch.float32, (n, B, q_len, H))
    _dev(status, "status", torch.int32, (1,))
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _dev(workspace, "workspace", torch.uint8)
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel()
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per request")
    _check("dcp_mla_decode_partial", load_library().dcp_mla_decode_partial(
        ctypes.byref(layout), shard_begin, shard_end, _ptr(q), B, q_len, H, _ptr(arena), pool_pages,
        _ptr(block_table), block_table.shape[1], max_pages, _ptr(seq_lens), float(scale), lse_base,
        _ptr(o_part), _dtype_code(o_part), _ptr(lse_part), ws_ptr, ws_bytes, _ptr(status), _stream(stream)))


def dcp_lse_merge(o_part, lse_part, lse_base, o, lse=None, stream=None):
    """Merge o_part [n, rows, 512] / lse_part [n, rows] into o [rows, 512] / lse [rows]."""
    n = o_part.shape[0]
    rows = o_part.numel() // (n * 512) if n else 0
    _dev(o_part, "o_part", o_part.dtype)
    if o_part.shape[-1] != 512:
        raise ValueError("o_part's last dim must be 512")
    _dev(lse_part, "lse_part", torch.float32)
    if lse_part.numel() != n * rows:
        raise ValueError("lse_part must hold n_parts * rows values")
    _dev(o, "o", o.dtype)
    if o.numel() != rows * 512:
        raise ValueError("o must hold rows * 512 values")
    if lse is not None:
        _dev(lse, "lse", torch.float32)
        if lse.numel() != rows:
            raise ValueError("lse must hold rows values")
    _check("dcp_lse_merge", load_library().dcp_lse_merge(
        n, rows, _ptr(o_part), _dtype_code(o_part), _ptr(lse_part), lse_base, _ptr(o), _dtype_code(o),
        _ptr(lse), _stream(stream)))


def dcp_mla_decode_static_scratch_bytes() -> int:
    """Bytes of the library's built-in scratch array (per device)."""
    return int(load_library().dcp_mla_decode_static_scratch_bytes())


def dcp_mla_decode_partial_static(layout, shard_begin, shard_end, q, arena, pool_pages, block_table, max_pages,
                                  seq_lens, scale, lse_base, o_part, lse_part, status, stream=None):
    """dcp_mla_decode_partial without a workspace, for callers that cannot allocate device memory.

    The library runs on its own built-in scratch array instead (one per device,
    held until exit).  Its first call on a device does a one-time address lookup,
    so make it before any stream capture; calls that overlap on the GPU share the
    array and must be ordered.
    """
    B, q_len, H, dk = q.shape
    n = shard_end - shard_begin
    _dev(q, "q", torch.bfloat16, (B, q_len, H, 576))
    _dev(arena, "arena", torch.bfloat16, (n, pool_pages * layout.page_size, 576))
    _dev(block_table, "block_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int64, (B,))
    _dev(o_part, "o_part", o_part.dtype, (n, B, q_len, H, 512))
    _dev(lse_part, "lse_part", torch.float32, (n, B, q_len, H))
    _dev(status, "status", torch.int32, (1,))
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per request")
    _check("dcp_mla_decode_partial_static", load_library().dcp_mla_decode_partial_static(
        ctypes.byref(layout), shard_begin, shard_end, _ptr(q), B, q_len, H, _ptr(arena), pool_pages,
        _ptr(block_table), block_table.shape[1], max_pages, _ptr(seq_lens), float(scale), lse_base,
        _ptr(o_part), _dtype_code(o_part), _ptr(lse_part), _ptr(status), _stream(stream)))


def _rows(t, name, width):
    """Row stride (elements) of a bf16 CUDA view [..., width] whose rows are equally strided."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be torch.bfloat16, got {t.dtype}")
    if t.shape[-1] != width or t.stride(-1) != 1:
        raise ValueError(f"{name} must be [..., {width}] with a contiguous last dim")
    row = t.stride(-2) if t.dim() >= 2 else width
    for i in range(t.dim() - 2):
        if t.shape[i + 1] > 1 and t.stride(i) != t.stride(i + 1) * t.shape[i + 1]:
            raise ValueError(f"{name}'s rows must be equally strided")
    return row


def dcp_absorb_q(q_nope, q_pe, w_kc, q, status=None, stream=None):
    """q [..., H, 576] = [q_nope @ w_kc[h] || q_pe] per head.

    q_nope [..., H, 128] and q_pe [..., H, 64] are bf16 views with a contiguous
    last dim and equally strided rows (slices of a [..., H, 192] q_b_proj output
    qualify); w_kc [H, 128, 512] bf16; q contiguous bf16."""
    H = w_kc.shape[0]
    _dev(w_kc, "w_kc", torch.bfloat16, (H, 128, 512))
    _dev(q, "q", torch.bfloat16)
    if q.dim() < 2 or q.shape[-1] != 576 or q.shape[-2] != H:
        raise ValueError(f"q must be [..., {H}, 576]")
    T = q.numel() // (H * 576)
    sn, sp = _rows(q_nope, "q_nope", 128), _rows(q_pe, "q_pe", 64)
    if q_nope.shape[:-1] != q.shape[:-1] or q_pe.shape[:-1] != q.shape[:-1]:
        raise ValueError("q_nope, q_pe and q must have the same leading dims")
    if status is not None:
        _dev(status, "status", torch.int32, (1,))
    _check("dcp_absorb_q", load_library().dcp_absorb_q(
        T, H, _ptr(q_nope), sn, _ptr(q_pe), sp, _ptr(w_kc), _ptr(q), _ptr(status), _stream(stream)))


def dcp_absorb_o(o, w_vc, v, status=None, stream=None):
    """v [..., H, 128] = o [..., H, 512] @ w_vc[h] per head (o, v f32 or bf16; w_vc [H, 512, 128] bf16)."""
    H = w_vc.shape[0]
    _dev(w_vc, "w_vc", torch.bfloat16, (H, 512, 128))
    _dev(o, "o", o.dtype)
    _dev(v, "v", v.dtype)
    if o.dim() < 2 or o.shape[-1] != 512 or o.shape[-2] != H:
        raise ValueError(f"o must be [..., {H}, 512]")
    if v.shape[:-1] != o.shape[:-1] or v.shape[-1] != 128:
        raise ValueError(f"v must be [..., {H}, 128] with o's leading dims")
    if status is not None:
        _dev(status, "status", torch.int32, (1,))
    T = o.numel() // (H * 512)
    _check("dcp_absorb_o", load_library().dcp_absorb_o(
        T, H, _ptr(o), _dtype_code(o), _ptr(w_vc), _ptr(v), _dtype_code(v), _ptr(status), _stream(stream)))


def dcp_lse_merge_absorb_o(o_part, lse_part, lse_base, w_vc, v, lse=None, status=None, stream=None):
    """v [..., H, 128] = bf16(LSE merge of o_part [n, ..., H, 512] / lse_part [n, ..., H]) @ w_vc[h];
    lse [..., H] gets the merged lse (optional).  One kernel; the merged o is not written."""
    n, H = o_part.shape[0], w_vc.shape[0]
    _dev(w_vc, "w_vc", torch.bfloat16, (H, 512, 128))
    _dev(o_part, "o_part", o_part.dtype)
    if o_part.shape[-1] != 512 or o_part.shape[-2] != H:
        raise ValueError(f"o_part must be [n, ..., {H}, 512]")
    T = o_part.numel() // (n * H * 512)
    _dev(lse_part, "lse_part", torch.float32)
    if lse_part.numel() != n * T * H:
        raise ValueError("lse_part must hold n * T * H values")
    _dev(v, "v", v.dtype)
    if v.numel() != T * H * 128 or v.shape[-1] != 128:
        raise ValueError("v must be [..., H, 128] with T * H rows")
    if lse is not None:
        _dev(lse, "lse", torch.float32)
        if lse.numel() != T * H:
            raise ValueError("lse must hold T * H values")
    if status is not None:
        _dev(status, "status", torch.int32, (1,))
    _check("dcp_lse_merge_absorb_o", load_library().dcp_lse_merge_absorb_o(
        n, T, H, _ptr(o_part), _dtype_code(o_part), _ptr(lse_part), lse_base, _ptr(w_vc), _ptr(v), _dtype_code(v),
        _ptr(lse), _ptr(status), _stream(stream)))


def dcp_a2a_chunk_bytes(n_held, T, H, world, wire_dtype=torch.bfloat16) -> int:
    """Bytes of one destination's chunk of an all-to-all buffer (see include/dcp.h)."""
    code = DCP_BF16 if wire_dtype == torch.bfloat16 else DCP_F32
    n = int(load_library().dcp_a2a_chunk_bytes(n_held, T, H, world, code))
    if n == 0:
        raise DcpError("dcp_a2a_chunk_bytes", DCP_ERR_INVALID, "invalid argument")
    return n


def dcp_pack_partials(o_part, lse_part, world, send, wire_dtype=torch.bfloat16, stream=None):
    """Pack o_part [n_held, ..., H, 512] / lse_part [n_held, ..., H] by head slice into
    send (uint8, [world, chunk]) for an all-to-all."""
    n_held, H = o_part.shape[0], o_part.shape[-2]
    T = o_part.numel() // (n_held * H * 512) if o_part.numel() else 0
    _dev(o_part, "o_part", o_part.dtype)
    if o_part.shape[-1] != 512:
        raise ValueError("o_part's last dim must be 512")
    _dev(lse_part, "lse_part", torch.float32)
    if lse_part.numel() != n_held * T * H:
        raise ValueError("lse_part must hold n_held * T * H values")
    chunk = dcp_a2a_chunk_bytes(n_held, T, H, world, wire_dtype)
    _dev(send, "send", torch.uint8)
    if send.numel() != world * chunk:
        raise ValueError(f"send must hold world * chunk = {world * chunk} bytes")
    code = DCP_BF16 if wire_dtype == torch.bfloat16 else DCP_F32
    _check("dcp_pack_partials", load_library().dcp_pack_partials(
        n_held, T, H, world, _ptr(o_part), _dtype_code(o_part), _ptr(lse_part), _ptr(send), code, _stream(stream)))


def dcp_lse_merge_packed(recv, world, n_held, lse_base, o, lse=None, wire_dtype=torch.bfloat16, stream=None):
    """Merge the world * n_held parts of an all-to-all receive buffer (uint8 [world, chunk])
    into o [rows, 512] (rows = T * H / world of this rank's heads) and lse [rows]."""
    rows = o.numel() // 512
    _dev(o, "o", o.dtype)
    if o.shape[-1] != 512:
        raise ValueError("o's last dim must be 512")
    _dev(recv, "recv", torch.uint8)
    code = DCP_BF16 if wire_dtype == torch.bfloat16 else DCP_F32
    if rows:
        e = 2 if code == DCP_BF16 else 4
        need = n_held * rows * (512 * e + 4)
        chunk = need + (-need % 256)
        if recv.numel() != world * chunk:
            raise ValueError(f"recv must hold world * chunk = {world * chunk} bytes")
    if lse is not None:
        _dev(lse, "lse", torch.float32)
        if lse.numel() != rows:
            raise ValueError("lse must hold rows values")
    _check("dcp_lse_merge_packed", load_library().dcp_lse_merge_packed(
        world, n_held, rows, _ptr(recv), code, lse_base, _ptr(o), _dtype_code(o), _ptr(lse), _stream(stream)))


def dcp_lse_rescale(lse_all, o_part, shard_begin, world, lse_base, o_sum, lse=None, stream=None):
    """AllGather + ReduceScatter, local step: lse_all [n_shards, ..., H] f32 (every shard),
    o_part [n_held, ..., H, 512] (this rank's shards) -> o_sum f32 [world, T, H / world, 512]
    (and lse f32 [world, T, H / world])."""
    n_shards, n_held, H = lse_all.shape[0], o_part.shape[0], o_part.shape[-2]
    T = o_part.numel() // (n_held * H * 512) if o_part.numel() else 0
    _dev(lse_all, "lse_all", torch.float32)
    if lse_all.numel() != n_shards * T * H:
        raise ValueError("lse_all must hold n_shards * T * H values")
    _dev(o_part, "o_part", o_part.dtype)
    _dev(o_sum, "o_sum", torch.float32)
    if o_sum.numel() != T * H * 512:
        raise ValueError("o_sum must hold T * H * 512 values")
    if lse is not None:
        _dev(lse, "lse", torch.float32)
        if lse.numel() != T * H:
            raise ValueError("lse must hold T * H values")
    _check("dcp_lse_rescale", load_library().dcp_lse_rescale(
        n_shards, shard_begin, n_held, T, H, world, _ptr(lse_all), _ptr(o_part), _dtype_code(o_part), lse_base,
        _ptr(o_sum), _ptr(lse), _stream(stream)))
