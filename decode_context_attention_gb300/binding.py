"""ctypes binding of libdcp_gb300.so (the C ABI in include/dcp.h).

Two layers, both argument marshalling only -- every byte of the merge is
computed by the CUDA kernels behind the C ABI:

* ``dcp_pack_send`` / ``dcp_lse_combine`` / ``dcp_unpack_combine`` /
  ``dcp_lse_pack_dim`` / ``dcp_status_string`` / ``dcp_last_error_message``:
  the C functions under their own names, taking raw integers (device
  addresses, sizes, element strides, a cudaStream_t handle).
* ``pack_send`` / ``lse_combine`` / ``unpack_combine``: the same calls taking
  torch CUDA tensors (views allowed); strides are read from the tensors and the
  kernels run on the current torch stream unless one is given.  Pinned host
  tensors are accepted too: the kernels then stream them over the host link
  (a pack that reads host inputs fuses the upload into the pack).

There is no fallback: if the library is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdcp_gb300.so")

DCP_OK = 0
DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.float8_e4m3fn: 3}
DCP_LSE_BASE_E, DCP_LSE_BASE_2 = 0, 1
DCP_SANITIZE_O, DCP_INPLACE_RANK0 = 1, 2
STATUS_NAMES = {0: "DCP_OK", 1: "DCP_ERR_INVALID_ARG", 2: "DCP_ERR_UNSUPPORTED_DTYPE",
                3: "DCP_ERR_HEADS_NOT_DIVISIBLE", 4: "DCP_ERR_MISALIGNED", 5: "DCP_ERR_ALIAS",
                6: "DCP_ERR_CUDA", 7: "DCP_ERR_TIMEOUT"}
# Every symbol include/dcp.h declares.
EXPORTS = ("dcp_lse_pack_dim", "dcp_status_string", "dcp_last_error_message", "dcp_pack_send",
           "dcp_lse_combine", "dcp_unpack_combine", "dcp_decode_attention_workspace_size",
           "dcp_decode_attention", "dcp_decode_attention_paged", "dcp_decode_attention_noalloc",
           "dcp_decode_attention_mla", "dcp_device_status")


class DcpError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.name}: {detail}")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m decode_context_attention_gb300.build` (no CPU fallback)")
        lib = ctypes.CDLL(path)
        i32, i64, vp, u32 = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint
        lib.dcp_lse_pack_dim.restype = i32
        lib.dcp_lse_pack_dim.argtypes = [i32]
        lib.dcp_status_string.restype = ctypes.c_char_p
        lib.dcp_status_string.argtypes = [i32]
        lib.dcp_last_error_message.restype = ctypes.c_char_p
        lib.dcp_last_error_message.argtypes = []
        lib.dcp_pack_send.restype = i32
        lib.dcp_pack_send.argtypes = ([i32] * 6 + [vp, i64, i64, i64] + [vp, i64, i64, i64]
                                      + [vp, i64, i64, i64, i64] + [vp, i64, i64, i64, i64] + [vp])
        merge_tail = [vp, i64, i64, i64] + [vp, i64, i64, i64] + [i32, i32, u32, vp]
        lib.dcp_lse_combine.restype = i32
        lib.dcp_lse_combine.argtypes = ([i32] * 6 + [vp, i64, i64, i64, i64]
                                        + [vp, i64, i64, i64, i64] + merge_tail)
        lib.dcp_unpack_combine.restype = i32
        lib.dcp_unpack_combine.argtypes = [i32] * 6 + [vp, i64, i64, i64, i64] + merge_tail
        lib.dcp_decode_attention_workspace_size.restype = ctypes.c_size_t
        lib.dcp_decode_attention_workspace_size.argtypes = [i32] * 6
        lib.dcp_decode_attention.restype = i32
        lib.dcp_decode_attention.argtypes = ([i32] * 6 + [vp, i64, i64] + [vp, i64, i64, i64, i64]
                                             + [vp, i64, i64, i64, i64] + [vp, i32, ctypes.c_float, i32]
                                             + [vp, i64, i64, i64] + [vp, i64, i64, i64]
                                             + [i32, vp, ctypes.c_size_t, vp])
        lib.dcp_decode_attention_paged.restype = i32
        lib.dcp_decode_attention_paged.argtypes = ([i32] * 6 + [vp, i64, i64] + [vp, i64, i64, i64, i64]
                                                   + [vp, i64, i64, i64, i64] + [i32, i32]
                                                   + [vp, i64, i64, i32]
                                                   + lib.dcp_decode_attention.argtypes[19:])
        lib.dcp_decode_attention_noalloc.restype = i32
        lib.dcp_decode_attention_noalloc.argtypes = lib.dcp_decode_attention.argtypes[:-3] + [vp]
        lib.dcp_decode_attention_mla.restype = i32
        lib.dcp_decode_attention_mla.argtypes = ([i32] * 6 + [vp, i64, i64] + [vp, i64, i64, i64]
                                                 + lib.dcp_decode_attention.argtypes[19:])
        lib.dcp_device_status.restype = i32
        lib.dcp_device_status.argtypes = []
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# raw C ABI, same names
# ---------------------------------------------------------------------------

def dcp_lse_pack_dim(dtype: int) -> int:
    return load().dcp_lse_pack_dim(dtype)


def dcp_status_string(status: int) -> str:
    return load().dcp_status_string(status).decode()


def dcp_last_error_message() -> str:
    return load().dcp_last_error_message().decode()


def dcp_pack_send(*args) -> int:
    return load().dcp_pack_send(*args)


def dcp_lse_combine(*args) -> int:
    return load().dcp_lse_combine(*args)


def dcp_unpack_combine(*args) -> int:
    return load().dcp_unpack_combine(*args)


def dcp_decode_attention_workspace_size(N: int, B: int, H: int, D: int, max_seq_len: int,
                                        split_tokens: int) -> int:
    return load().dcp_decode_attention_workspace_size(N, B, H, D, max_seq_len, split_tokens)


def dcp_decode_attention(*args) -> int:
    return load().dcp_decode_attention(*args)


def dcp_decode_attention_mla(*args) -> int:
    return load().dcp_decode_attention_mla(*args)


def dcp_device_status() -> int:
    return load().dcp_device_status()


def check(status: int, where: str) -> None:
    if status != DCP_OK:
        raise DcpError(status, where, dcp_last_error_message() or dcp_status_string(status))


# ---------------------------------------------------------------------------
# torch-tensor layer
# ---------------------------------------------------------------------------

def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in DTYPE_CODES:
        raise DcpError(2, "dtype", f"unsupported payload dtype {t.dtype}")
    return DTYPE_CODES[t.dtype]


def _need_cuda(*ts):
    """Operands must be reachable by the kernels: CUDA tensors, or page-locked
    (pinned) host tensors, which the kernels read and write in place over the
    host link.  Ordinary host tensors are refused (there is no CPU fallback)."""
    for t in ts:
        if t is not None and not (t.is_cuda or t.is_pinned()):
            raise ValueError("DCP kernels take CUDA tensors or pinned host tensors (no CPU fallback)")


def _lead(t: torch.Tensor, nd: int) -> torch.Tensor:
    """Add a leading group axis of size 1 if `t` has nd - 1 dims."""
    if t.dim() == nd - 1:
        return t.unsqueeze(0)
    if t.dim() != nd:
        raise ValueError(f"expected a {nd - 1}- or {nd}-dim tensor, got shape {tuple(t.shape)}")
    return t


def _inner_ok(t: torch.Tensor) -> None:
    if t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError("the innermost (D) dimension must have stride 1")


class _Prepared:
    """One entry-point call with its arguments marshalled once; calling it
    enqueues the kernel again (same tensors, same stream) and checks the status."""

    def __init__(self, fn_name: str, args: tuple, keep: tuple):
        self._fn = getattr(load(), fn_name)
        self._name = fn_name
        self._args = args
        self._keep = keep  # keeps the tensors (and so their memory) alive

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != DCP_OK:
            check(st, self._name)


def prepare_pack_send(o: torch.Tensor, lse: torch.Tensor, dst_o: torch.Tensor,
                      dst_lse: torch.Tensor, stream=None) -> _Prepared:
    """O [G,]B,H,D and LSE [G,]B,H -> dst_o [G,]N,B,H/N,D and dst_lse [G,]N,B,H/N (views)."""
    _need_cuda(o, lse, dst_o, dst_lse)
    o4, l3, d5, dl4 = _lead(o, 4), _lead(lse, 3), _lead(dst_o, 5), _lead(dst_lse, 4)
    _inner_ok(o4)
    _inner_ok(d5)
    if lse.dtype != torch.float32 or dst_lse.dtype != torch.float32:
        raise ValueError("LSE tensors are fp32")
    if dst_o.dtype != o.dtype:
        raise ValueError("dst_o must have the payload dtype of o")
    G, B, H, D = o4.shape
    N = d5.shape[1]
    args = (_dtype_code(o), N, B, H, D, G,
            o4.data_ptr(), o4.stride(0), o4.stride(1), o4.stride(2),
            l3.data_ptr(), l3.stride(0), l3.stride(1), l3.stride(2),
            d5.data_ptr(), d5.stride(0), d5.stride(1), d5.stride(2), d5.stride(3),
            dl4.data_ptr(), dl4.stride(0), dl4.stride(1), dl4.stride(2), dl4.stride(3),
            _stream_handle(stream))
    return _Prepared("dcp_pack_send", args, (o, lse, dst_o, dst_lse))


def _base_code(base: str) -> int:
    return {"e": DCP_LSE_BASE_E, "2": DCP_LSE_BASE_2}[str(base)]


def _out_lse_args(out_lse):
    if out_lse is None:
        return (None, 0, 0, 0)
    ul3 = _lead(out_lse, 3)
    return (ul3.data_ptr(), ul3.stride(0), ul3.stride(1), ul3.stride(2))


def prepare_lse_combine(o: torch.Tensor, lse: torch.Tensor, out: torch.Tensor,
                        out_lse: torch.Tensor | None = None, base: str = "e",
                        sanitize: bool = False, inplace: bool = False, stream=None) -> _Prepared:
    """Merge O [G,]N,B,Hc,D with LSE [G,]N,B,Hc into out [G,]B,Hc,D (+ out_lse [G,]B,Hc)."""
    _need_cuda(o, lse, out, out_lse)
    o5, l4, u4 = _lead(o, 5), _lead(lse, 4), _lead(out, 4)
    _inner_ok(o5)
    _inner_ok(u4)
    G, N, B, Hc, D = o5.shape
    flags = (DCP_SANITIZE_O if sanitize else 0) | (DCP_INPLACE_RANK0 if inplace else 0)
    args = (_dtype_code(o), N, B, Hc, D, G,
            o5.data_ptr(), o5.stride(0), o5.stride(1), o5.stride(2), o5.stride(3),
            l4.data_ptr(), l4.stride(0), l4.stride(1), l4.stride(2), l4.stride(3),
            u4.data_ptr(), u4.stride(0), u4.stride(1), u4.stride(2),
            *_out_lse_args(out_lse), _base_code(base), 1 if out_lse is not None else 0, flags,
            _stream_handle(stream))
    return _Prepared("dcp_lse_combine", args, (o, lse, out, out_lse))


def prepare_unpack_combine(recv: torch.Tensor, D: int, out: torch.Tensor,
                           out_lse: torch.Tensor | None = None, base: str = "e",
                           sanitize: bool = False, stream=None) -> _Prepared:
    """Merge the interleaved receive rows recv [G,]N,B,Hpr,D+lpd into out [G,]B,Hpr,D."""
    _need_cuda(recv, out, out_lse)
    r5, u4 = _lead(recv, 5), _lead(out, 4)
    _inner_ok(r5)
    _inner_ok(u4)
    G, N, B, Hpr, _ = r5.shape
    args = (_dtype_code(recv), N, B, Hpr, D, G,
            r5.data_ptr(), r5.stride(0), r5.stride(1), r5.stride(2), r5.stride(3),
            u4.data_ptr(), u4.stride(0), u4.stride(1), u4.stride(2),
            *_out_lse_args(out_lse), _base_code(base), 1 if out_lse is not None else 0,
            DCP_SANITIZE_O if sanitize else 0, _stream_handle(stream))
    return _Prepared("dcp_unpack_combine", args, (recv, out, out_lse))


def pack_send(o, lse, dst_o, dst_lse, stream=None) -> None:
    prepare_pack_send(o, lse, dst_o, dst_lse, stream)()


def lse_combine(o, lse, out, out_lse=None, base="e", sanitize=False, inplace=False,
                stream=None) -> None:
    prepare_lse_combine(o, lse, out, out_lse, base, sanitize, inplace, stream)()


def unpack_combine(recv, D, out, out_lse=None, base="e", sanitize=False, stream=None) -> None:
    prepare_unpack_combine(recv, D, out, out_lse, base, sanitize, stream)()


def _default_workspace(workspace, device, N, B, H, D, max_seq_len, split_tokens):
    """The caller's workspace, else a fresh one of the size the call needs."""
    if workspace is not None:
        return workspace
    nbytes = dcp_decode_attention_workspace_size(N, B, H, D, int(max_seq_len), int(split_tokens))
    return torch.empty(nbytes, dtype=torch.uint8, device=device) if nbytes else None


def prepare_decode_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                             max_seq_len: int, o: torch.Tensor, lse: torch.Tensor, sm_scale: float,
                             base: str = "e", split_tokens: int = 1024,
                             workspace: torch.Tensor | None = None, stream=None) -> _Prepared:
    """Each rank's decode attention over its round-robin share of the KV cache.

    q [B,H,D]; k, v [N,B,Lc,Hkv,D] local caches (token i of rank r = global
    token i*N + r); seq_lens [B] int32 global lengths; o [N,B,H,D], lse [N,B,H].
    `workspace` (uint8, device, workspace_bytes() long): the split partials and
    the work counters; allocated here when not given."""
    _need_cuda(q, k, v, seq_lens, o, lse, workspace)
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    for t in (q, k, v, o):
        _inner_ok(t)
    B, H, D = q.shape
    N, _, _, Hkv, _ = k.shape
    workspace = _default_workspace(workspace, q.device, N, B, H, D, max_seq_len, split_tokens)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_dtype_code(q), N, B, H, Hkv, D,
            q.data_ptr(), q.stride(0), q.stride(1),
            k.data_ptr(), k.stride(0), k.stride(1), k.stride(2), k.stride(3),
            v.data_ptr(), v.stride(0), v.stride(1), v.stride(2), v.stride(3),
            seq_lens.data_ptr(), int(max_seq_len), float(sm_scale), int(split_tokens),
            o.data_ptr(), o.stride(0), o.stride(1), o.stride(2),
            lse.data_ptr(), lse.stride(0), lse.stride(1), lse.stride(2),
            _base_code(base), None if workspace is None else workspace.data_ptr(), ws_bytes,
            _stream_handle(stream))
    return _Prepared("dcp_decode_attention", args, (q, k, v, seq_lens, o, lse, workspace))


def prepare_decode_attention_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                                   block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                                   o: torch.Tensor, lse: torch.Tensor, sm_scale: float, base: str = "e",
                                   split_tokens: int = 1024, workspace: torch.Tensor | None = None,
                                   stream=None) -> _Prepared:
    """prepare_decode_attention over paged caches: k_pages, v_pages
    [N, num_pages, page_size, Hkv, D]; block_table [N, B, max_pages] int32, local
    token i of request b on rank r in slot i % page_size of page
    block_table[r, b, i // page_size]."""
    _need_cuda(q, k_pages, v_pages, block_table, seq_lens, o, lse, workspace)
    if seq_lens.dtype != torch.int32 or block_table.dtype != torch.int32:
        raise ValueError("seq_lens and block_table must be int32")
    if block_table.dim() != 3 or block_table.shape[-1] > 1 and block_table.stride(-1) != 1:
        raise ValueError("block_table is [N, B, max_pages] with unit stride along the pages")
    for t in (q, k_pages, v_pages, o):
        _inner_ok(t)
    B, H, D = q.shape
    N, num_pages, page_size, Hkv, _ = k_pages.shape
    workspace = _default_workspace(workspace, q.device, N, B, H, D, max_seq_len, split_tokens)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_dtype_code(q), N, B, H, Hkv, D,
            q.data_ptr(), q.stride(0), q.stride(1),
            k_pages.data_ptr(), k_pages.stride(0), k_pages.stride(1), k_pages.stride(2), k_pages.stride(3),
            v_pages.data_ptr(), v_pages.stride(0), v_pages.stride(1), v_pages.stride(2), v_pages.stride(3),
            num_pages, page_size,
            block_table.data_ptr(), block_table.stride(0), block_table.stride(1), block_table.shape[2],
            seq_lens.data_ptr(), int(max_seq_len), float(sm_scale), int(split_tokens),
            o.data_ptr(), o.stride(0), o.stride(1), o.stride(2),
            lse.data_ptr(), lse.stride(0), lse.stride(1), lse.stride(2),
            _base_code(base), None if workspace is None else workspace.data_ptr(), ws_bytes,
            _stream_handle(stream))
    return _Prepared("dcp_decode_attention_paged", args,
                     (q, k_pages, v_pages, block_table, seq_lens, o, lse, workspace))


def decode_attention_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len, o, lse, sm_scale, base="e",
                           split_tokens=1024, workspace=None, stream=None) -> None:
    prepare_decode_attention_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len, o, lse, sm_scale,
                                   base, split_tokens, workspace, stream)()


def decode_attention(q, k, v, seq_lens, max_seq_len, o, lse, sm_scale, base="e", split_tokens=1024,
                     workspace=None, stream=None) -> None:
    prepare_decode_attention(q, k, v, seq_lens, max_seq_len, o, lse, sm_scale, base, split_tokens,
                             workspace, stream)()


def prepare_decode_attention_mla(q: torch.Tensor, kv: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                                 o: torch.Tensor, lse: torch.Tensor, sm_scale: float, base: str = "2",
                                 split_tokens: int = 1024, workspace: torch.Tensor | None = None,
                                 stream=None) -> _Prepared:
    """Each rank's decode attention over its round-robin share of an
    absorbed-MLA latent cache.

    q [B,H,Dk]; kv [N,B,Lc,Dk] latent caches (the value is each row's first
    Dv = o.shape[-1] elements); seq_lens [B] int32 global lengths;
    o [N,B,H,Dv], lse [N,B,H].  `workspace` as for prepare_decode_attention,
    sized workspace_bytes(N, B, H, Dv, max_seq_len, split_tokens)."""
    _need_cuda(q, kv, seq_lens, o, lse, workspace)
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    for t in (q, kv, o):
        _inner_ok(t)
    B, H, Dk = q.shape
    N = kv.shape[0]
    Dv = o.shape[-1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_dtype_code(q), N, B, H, Dk, Dv,
            q.data_ptr(), q.stride(0), q.stride(1),
            kv.data_ptr(), kv.stride(0), kv.stride(1), kv.stride(2),
            seq_lens.data_ptr(), int(max_seq_len), float(sm_scale), int(split_tokens),
            o.data_ptr(), o.stride(0), o.stride(1), o.stride(2),
            lse.data_ptr(), lse.stride(0), lse.stride(1), lse.stride(2),
            _base_code(base), None if workspace is None else workspace.data_ptr(), ws_bytes,
            _stream_handle(stream))
    return _Prepared("dcp_decode_attention_mla", args, (q, kv, seq_lens, o, lse, workspace))


def decode_attention_mla(q, kv, seq_lens, max_seq_len, o, lse, sm_scale, base="2", split_tokens=1024,
                         workspace=None, stream=None) -> None:
    prepare_decode_attention_mla(q, kv, seq_lens, max_seq_len, o, lse, sm_scale, base, split_tokens,
                                 workspace, stream)()


def device_status() -> int:
    """dcp_device_status(): 0, or DCP_ERR_TIMEOUT when a tensor-core kernel
    gave up on a bounded wait since the last call (synchronises)."""
    return load().dcp_device_status()


def workspace_bytes(N: int, B: int, H: int, D: int, max_seq_len: int, split_tokens: int) -> int:
    return dcp_decode_attention_workspace_size(N, B, H, D, max_seq_len, split_tokens)
