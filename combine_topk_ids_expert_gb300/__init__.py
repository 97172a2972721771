"""GB300-native MoE expert-parallel token dispatch and combine.

A thin binding over libep_gb300.so (the C ABI of include/ep.h). Every step of
the dispatch/combine path runs in the library's CUDA kernels; this module only
marshals arguments. PyTorch supplies device memory (the workspace and the
caller's tensors) and streams.

Module-level functions carry the C names (``ep_dispatch``, ``ep_combine``,
...) and take a buffer handle and torch tensors. ``Buffer`` wraps them for
everyday use and returns torch views into the workspace::

    buf = Buffer(num_max_tokens_per_rank=8192, hidden=7168, num_experts=256,
                 num_ranks=8, topk=8, dtype=torch.bfloat16)
    d = buf.dispatch(x_TD, topk_scores_TK, topk_expert_ids_TK, num_tokens_per_rank=8192)
    y = experts(d.recv_x)                    # [R, S, D], rows past each rank's total undefined
    out_TD = buf.combine(y, topk_scores_TK)  # [T, D]
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import torch

from . import _abi
from ._abi import (EP_BF16, EP_DEVERR_BAD_ID, EP_DEVERR_DEBUG_STRAY, EP_DEVERR_DEBUG_UNWRITTEN,
                   EP_DEVERR_ROW_OOB, EP_DEVERR_TIMEOUT, EP_F32, EP_NOALLOC_SCRATCH_BYTES,
                   EP_LAYOUT_PACKED, EP_LAYOUT_STRIDED, EP_PERMUTE_BULK, EP_PERMUTE_DEFAULT,
                   EP_PERMUTE_VEC, EpBufferInfo, EpConfig, EpDedupOut, EpDispatchOut, EpError,
                   EpLayout, check)

__all__ = [
    "Buffer", "Layout", "DispatchResult", "EpConfig", "EpError",
    "ep_buffer_required_bytes", "ep_buffer_init", "ep_buffer_destroy", "ep_dispatch_layout",
    "ep_dispatch", "ep_dispatch_permute", "ep_combine", "ep_combine_backward",
    "ep_dispatch_backward", "ep_dispatch_dedup", "ep_dedup_expand", "ep_expert_gemm",
    "ep_get_device_error", "DedupResult",
    "ep_buffer_query", "ep_dispatch_layout_noalloc", "ep_dispatch_layout_noalloc_scratch_bytes",
    "EP_NOALLOC_SCRATCH_BYTES", "ep_pattern_probe", "ep_pad_tokens", "group_num_tokens_per_rank",
    "ep_derive_max_tokens_pretrain",
    "ep_derive_max_tokens_inference", "ep_validate_max_tokens", "ep_status_string",
    "EP_BF16", "EP_F32", "EP_PERMUTE_DEFAULT", "EP_PERMUTE_VEC", "EP_PERMUTE_BULK",
    "EP_LAYOUT_STRIDED", "EP_LAYOUT_PACKED",
    "EP_DEVERR_BAD_ID", "EP_DEVERR_ROW_OOB", "EP_DEVERR_TIMEOUT", "EP_DEVERR_DEBUG_UNWRITTEN",
    "EP_DEVERR_DEBUG_STRAY", "library_path",
]

_TORCH_TO_EP = {torch.bfloat16: EP_BF16, torch.float32: EP_F32}
_EP_TO_TORCH = {EP_BF16: torch.bfloat16, EP_F32: torch.float32}


def library_path() -> str:
    return _abi.LIB_PATH


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check_dtype(t: torch.Tensor, dtype: torch.dtype, name: str) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


# ---------------------------------------------------------------------------
# C-named functions (one call each)
# ---------------------------------------------------------------------------

def ep_buffer_required_bytes(cfg: EpConfig) -> int:
    return int(_abi.lib().ep_buffer_required_bytes(C.byref(cfg)))


def ep_buffer_init(cfg: EpConfig, workspace: torch.Tensor) -> C.c_void_p:
    h = C.c_void_p()
    check(_abi.lib().ep_buffer_init(C.byref(cfg), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), C.byref(h)),
          "ep_buffer_init")
    return h


def ep_buffer_destroy(handle) -> None:
    check(_abi.lib().ep_buffer_destroy(handle), "ep_buffer_destroy")


def ep_dispatch_layout(handle, topk_expert_ids_TK: torch.Tensor, num_tokens: int,
                       num_tokens_per_rank: int, stream=None,
                       host_tokens_per_expert: torch.Tensor | None = None) -> EpLayout:
    _check_dtype(topk_expert_ids_TK, torch.int32, "topk_expert_ids_TK")
    host = None
    if host_tokens_per_expert is not None:
        _check_dtype(host_tokens_per_expert, torch.int32, "host_tokens_per_expert")
        if host_tokens_per_expert.is_cuda or not host_tokens_per_expert.is_contiguous():
            raise ValueError("host_tokens_per_expert must be a contiguous CPU tensor")
        host = host_tokens_per_expert.data_ptr()
    out = EpLayout()
    check(_abi.lib().ep_dispatch_layout(handle, _ptr(topk_expert_ids_TK), num_tokens,
                                        num_tokens_per_rank, _stream(stream), C.byref(out), host),
          "ep_dispatch_layout")
    return out


def ep_dispatch(handle, x_TD: torch.Tensor, topk_scores_TK: torch.Tensor,
                topk_expert_ids_TK: torch.Tensor, num_tokens: int, num_tokens_per_rank: int,
                stream=None) -> EpDispatchOut:
    _check_dtype(topk_scores_TK, torch.float32, "topk_scores_TK")
    _check_dtype(topk_expert_ids_TK, torch.int32, "topk_expert_ids_TK")
    out = EpDispatchOut()
    check(_abi.lib().ep_dispatch(handle, _ptr(x_TD), _ptr(topk_scores_TK),
                                 _ptr(topk_expert_ids_TK), num_tokens, num_tokens_per_rank,
                                 _stream(stream), C.byref(out)), "ep_dispatch")
    return out


def ep_dispatch_permute(handle, x_TD: torch.Tensor, topk_scores_TK: torch.Tensor,
                        stream=None) -> EpDispatchOut:
    _check_dtype(topk_scores_TK, torch.float32, "topk_scores_TK")
    out = EpDispatchOut()
    check(_abi.lib().ep_dispatch_permute(handle, _ptr(x_TD), _ptr(topk_scores_TK),
                                         _stream(stream), C.byref(out)), "ep_dispatch_permute")
    return out


def ep_combine(handle, y_recv: torch.Tensor, topk_scores_TK: torch.Tensor, num_tokens: int,
               out_TD: torch.Tensor, out_dtype: int, stream=None) -> None:
    _check_dtype(topk_scores_TK, torch.float32, "topk_scores_TK")
    check(_abi.lib().ep_combine(handle, _ptr(y_recv), _ptr(topk_scores_TK), num_tokens,
                                _ptr(out_TD), out_dtype, _stream(stream)), "ep_combine")


def ep_combine_backward(handle, grad_out_TD: torch.Tensor, y_recv: torch.Tensor | None,
                        topk_scores_TK: torch.Tensor, num_tokens: int, grad_y_recv: torch.Tensor,
                        grad_scores_TK: torch.Tensor | None = None, stream=None) -> None:
    _check_dtype(topk_scores_TK, torch.float32, "topk_scores_TK")
    if grad_scores_TK is not None:
        _check_dtype(grad_scores_TK, torch.float32, "grad_scores_TK")
    check(_abi.lib().ep_combine_backward(handle, _ptr(grad_out_TD), _ptr(y_recv),
                                         _ptr(topk_scores_TK), num_tokens, _ptr(grad_y_recv),
                                         _ptr(grad_scores_TK), _stream(stream)),
          "ep_combine_backward")


def ep_dispatch_backward(handle, grad_recv_x: torch.Tensor,
                         grad_recv_scores: torch.Tensor | None, num_tokens: int,
                         grad_x_TD: torch.Tensor, grad_x_dtype: int,
                         grad_scores_TK: torch.Tensor | None = None, stream=None) -> None:
    for name, t in (("grad_recv_scores", grad_recv_scores), ("grad_scores_TK", grad_scores_TK)):
        if t is not None:
            _check_dtype(t, torch.float32, name)
    check(_abi.lib().ep_dispatch_backward(handle, _ptr(grad_recv_x), _ptr(grad_recv_scores),
                                          num_tokens, _ptr(grad_x_TD), grad_x_dtype,
                                          _ptr(grad_scores_TK), _stream(stream)),
          "ep_dispatch_backward")


def ep_dispatch_dedup(handle, x_TD: torch.Tensor, topk_scores_TK: torch.Tensor,
                      topk_expert_ids_TK: torch.Tensor, num_tokens: int, num_tokens_per_rank: int,
                      stream=None) -> EpDedupOut:
    _check_dtype(topk_scores_TK, torch.float32, "topk_scores_TK")
    _check_dtype(topk_expert_ids_TK, torch.int32, "topk_expert_ids_TK")
    out = EpDedupOut()
    check(_abi.lib().ep_dispatch_dedup(handle, _ptr(x_TD), _ptr(topk_scores_TK),
                                       _ptr(topk_expert_ids_TK), num_tokens, num_tokens_per_rank,
                                       _stream(stream), C.byref(out)), "ep_dispatch_dedup")
    return out


def ep_dedup_expand(handle, topk_expert_ids_TK: torch.Tensor, y_recv: torch.Tensor,
                    stream=None) -> None:
    _check_dtype(topk_expert_ids_TK, torch.int32, "topk_expert_ids_TK")
    check(_abi.lib().ep_dedup_expand(handle, _ptr(topk_expert_ids_TK), _ptr(y_recv),
                                     _stream(stream)), "ep_dedup_expand")


def ep_expert_gemm(handle, x_recv: torch.Tensor, weights: torch.Tensor, din: int, dout: int,
                   y_recv: torch.Tensor, stream=None) -> None:
    for name, t in (("x_recv", x_recv), ("weights", weights), ("y_recv", y_recv)):
        _check_dtype(t, torch.bfloat16, name)
    check(_abi.lib().ep_expert_gemm(handle, _ptr(x_recv), _ptr(weights), din, dout, _ptr(y_recv),
                                    _stream(stream)), "ep_expert_gemm")


def ep_get_device_error(handle, stream=None) -> int:
    v = C.c_uint32(0)
    check(_abi.lib().ep_get_device_error(handle, _stream(stream), C.byref(v)),
          "ep_get_device_error")
    return int(v.value)


def ep_buffer_query(handle) -> EpBufferInfo:
    info = EpBufferInfo()
    check(_abi.lib().ep_buffer_query(handle, C.byref(info)), "ep_buffer_query")
    return info


def ep_dispatch_layout_noalloc(topk_expert_ids_TK: torch.Tensor, num_tokens: int,
                               num_tokens_per_rank: int, topk: int, num_experts: int,
                               num_ranks: int, tokens_per_expert: torch.Tensor,
                               expert_offset: torch.Tensor, rows_per_rank: torch.Tensor,
                               rank_prefix: torch.Tensor, tokens_in_rank: torch.Tensor,
                               pos: torch.Tensor, error_flags: torch.Tensor | None = None,
                               stream=None) -> None:
    """The layout without a buffer, for callers that cannot allocate device
    memory: the caller supplies every output tensor (int32, on one CUDA device);
    the library uses its own fixed device scratch and allocates nothing. The
    tensors' sizes are checked here, since the C call only sees pointers: ids
    and pos hold num_tokens * topk entries, the per-expert outputs num_experts,
    the per-rank outputs num_ranks, error_flags (optional) one word."""
    T, K, E, R = int(num_tokens), int(topk), int(num_experts), int(num_ranks)
    if T < 0 or int(num_tokens_per_rank) < T:
        raise ValueError(f"need 0 <= num_tokens ({T}) <= num_tokens_per_rank "
                         f"({num_tokens_per_rank})")
    tensors = [("topk_expert_ids_TK", topk_expert_ids_TK, T * K),
               ("tokens_per_expert", tokens_per_expert, E), ("expert_offset", expert_offset, E),
               ("rows_per_rank", rows_per_rank, R), ("rank_prefix", rank_prefix, R),
               ("tokens_in_rank", tokens_in_rank, R), ("pos", pos, T * K)]
    if error_flags is not None:
        tensors.append(("error_flags", error_flags, 1))
    device = topk_expert_ids_TK.device
    if not topk_expert_ids_TK.is_cuda:
        raise ValueError("topk_expert_ids_TK must be a CUDA tensor")
    for name, t, n in tensors:
        if name != "error_flags":
            _check_dtype(t, torch.int32, name)
        elif t.dtype not in (torch.int32, torch.uint32) or not t.is_cuda or not t.is_contiguous():
            raise TypeError("error_flags must be a contiguous 4-byte integer CUDA tensor")
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, topk_expert_ids_TK on {device}")
        if t.numel() < n:
            raise ValueError(f"{name} has {t.numel()} elements, the call needs {n}")
    with torch.cuda.device(device):     # the device whose scratch the call uses
        check(_abi.lib().ep_dispatch_layout_noalloc(
            _ptr(topk_expert_ids_TK), T, num_tokens_per_rank, K, E, R, _ptr(tokens_per_expert),
            _ptr(expert_offset), _ptr(rows_per_rank), _ptr(rank_prefix), _ptr(tokens_in_rank),
            _ptr(pos), _ptr(error_flags), _stream(stream)), "ep_dispatch_layout_noalloc")


def ep_dispatch_layout_noalloc_scratch_bytes(num_tokens: int, topk: int, num_experts: int,
                                             num_ranks: int) -> int:
    """Bytes of the fixed device scratch that ep_dispatch_layout_noalloc needs for
    these sizes (host arithmetic only); accepted when <= EP_NOALLOC_SCRATCH_BYTES."""
    return int(_abi.lib().ep_dispatch_layout_noalloc_scratch_bytes(num_tokens, topk,
                                                                   num_experts, num_ranks))


def ep_pattern_probe(pattern: int, src: torch.Tensor | None, dst: torch.Tensor, rows: int,
                     row_bytes: int, fan: int = 1, stream=None) -> None:
    """Measurement aid: one of the hot path's HBM access patterns (EP_PATTERN_*)
    on `rows` rows of row_bytes, alone in a kernel. Sizes are checked here:
    FANOUT writes fan*rows rows, GATHER reads fan*rows rows, READ writes one
    16-byte word per row."""
    n_src = rows * row_bytes * (fan if pattern == _abi.EP_PATTERN_GATHER else 1)
    n_dst = (rows * 16 if pattern == _abi.EP_PATTERN_READ
             else rows * row_bytes * (fan if pattern == _abi.EP_PATTERN_FANOUT else 1))
    if pattern != _abi.EP_PATTERN_WRITE and (src is None or src.numel() * src.element_size() < n_src):
        raise ValueError(f"src must hold {n_src} bytes")
    if dst.numel() * dst.element_size() < n_dst:
        raise ValueError(f"dst must hold {n_dst} bytes")
    check(_abi.lib().ep_pattern_probe(pattern, _ptr(src), _ptr(dst), rows, row_bytes, fan,
                                      _stream(stream)), "ep_pattern_probe")


def ep_pad_tokens(n: int) -> int:
    return int(_abi.lib().ep_pad_tokens(n))


def group_num_tokens_per_rank(num_local_tokens: int, group=None) -> int:
    """num_tokens_per_rank for one expert-parallel group: the largest token count
    of its ranks ("fix(moe): equalize and align per-rank token counts for HybridEP
    dispatch", section "Fix": every rank pads to the EP-group max; dispatch then
    rounds it up to a multiple of 4, as ep_pad_tokens shows). One all-reduce (MAX)
    over the torch.distributed `group`, on a CUDA tensor under NCCL and a host
    tensor otherwise; without an initialised process group, the local count.
    Host logic on host integers: nothing here reads device memory."""
    import torch.distributed as dist
    n = int(num_local_tokens)
    if n < 0:
        raise ValueError(f"num_local_tokens must be >= 0, got {n}")
    if not (dist.is_available() and dist.is_initialized()):
        return n
    nccl = dist.get_backend(group) == "nccl"
    dev = torch.device("cuda", torch.cuda.current_device()) if nccl else torch.device("cpu")
    t = torch.tensor([n], dtype=torch.int64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return int(t.item())


def ep_derive_max_tokens_pretrain(local_batch_size: int, seq_len: int, cp: int, tp: int) -> int:
    return int(_abi.lib().ep_derive_max_tokens_pretrain(local_batch_size, seq_len, cp, tp))


def ep_derive_max_tokens_inference(max_num_batched_tokens: int, cp: int, tp: int) -> int:
    return int(_abi.lib().ep_derive_max_tokens_inference(max_num_batched_tokens, cp, tp))


def ep_validate_max_tokens(configured: int, derived: int) -> int:
    return int(_abi.lib().ep_validate_max_tokens(configured, derived))


def ep_status_string(status: int) -> str:
    return _abi.lib().ep_status_string(status).decode()


# ---------------------------------------------------------------------------
# Buffer: workspace ownership plus torch views of the results
# ---------------------------------------------------------------------------

@dataclass
class Layout:
    tokens_per_expert: torch.Tensor   # [E] int32
    expert_offset: torch.Tensor       # [E] int32
    rows_per_rank: torch.Tensor       # [R] int32
    rank_prefix: torch.Tensor         # [R] int32, inclusive
    tokens_in_rank: torch.Tensor      # [R] int32
    pos: torch.Tensor                 # [T, K] int32
    num_tokens: int
    padded_tokens: int
    rank_stride: int
    packed: bool


@dataclass
class DispatchResult:
    recv_x: torch.Tensor              # [R, S, D] (strided) or [R*S, D] (packed)
    recv_scores: torch.Tensor         # [R, S] or [R*S] fp32
    recv_src: torch.Tensor            # [R, S] or [R*S] int32
    layout: Layout


@dataclass
class DedupResult:
    recv_x: torch.Tensor              # [R, P, D]: one row per distinct (token, rank)
    recv_tok_src: torch.Tensor        # [R, P] int32 source token
    recv_topk_idx: torch.Tensor       # [R, P, K] int32 local expert index or -1
    recv_topk_w: torch.Tensor         # [R, P, K] fp32 score or 0
    tok_pos: torch.Tensor             # [T, R] int32 row of (t, r) or -1
    layout: Layout                    # tokens_in_rank[r] = rank r's rows


class Buffer:
    """A dispatcher buffer: one workspace sized from num_max_tokens_per_rank,
    reused by every call (no allocation after construction)."""

    def __init__(self, num_max_tokens_per_rank: int, hidden: int, num_experts: int,
                 num_ranks: int, topk: int, dtype: torch.dtype = torch.bfloat16,
                 num_sms: int = 0, permute_impl: int = EP_PERMUTE_DEFAULT, device=None,
                 layout: str = "strided"):
        if dtype not in _TORCH_TO_EP:
            raise TypeError(f"dtype must be bfloat16 or float32, got {dtype}")
        mode = {"strided": EP_LAYOUT_STRIDED, "packed": EP_LAYOUT_PACKED}[layout]
        self.cfg = EpConfig(num_max_tokens_per_rank, hidden, num_experts, num_ranks, topk,
                            _TORCH_TO_EP[dtype], num_sms, permute_impl, mode)
        self.packed = mode == EP_LAYOUT_PACKED
        nbytes = ep_buffer_required_bytes(self.cfg)
        if nbytes == 0:
            raise EpError(_abi.EP_ERR_INVALID_ARG, "ep_buffer_required_bytes")
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        self.device = dev
        self.dtype = dtype
        self.E, self.R, self.K, self.D = num_experts, num_ranks, topk, hidden
        with torch.cuda.device(dev):
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            self.handle = ep_buffer_init(self.cfg, self.workspace)
        self._base = self.workspace.data_ptr()

    # -- views -------------------------------------------------------------
    def _view(self, ptr: int, dtype: torch.dtype, shape: tuple) -> torch.Tensor:
        n = 1
        for s in shape:
            n *= s
        esize = torch.empty((), dtype=dtype).element_size()
        off = ptr - self._base
        return self.workspace[off:off + n * esize].view(dtype).view(*shape)

    def _layout(self, L: EpLayout) -> Layout:
        T, E, R, K = L.num_tokens, self.E, self.R, self.K
        self._stride = L.rank_stride
        i32 = torch.int32
        return Layout(
            tokens_per_expert=self._view(L.tokens_per_expert, i32, (E,)),
            expert_offset=self._view(L.expert_offset, i32, (E,)),
            rows_per_rank=self._view(L.rows_per_rank, i32, (R,)),
            rank_prefix=self._view(L.rank_prefix, i32, (R,)),
            tokens_in_rank=self._view(L.tokens_in_rank, i32, (R,)),
            pos=self._view(L.pos, i32, (T, K)),
            num_tokens=T, padded_tokens=L.padded_tokens, rank_stride=L.rank_stride,
            packed=bool(L.packed))

    def _dispatch_result(self, d: EpDispatchOut) -> DispatchResult:
        S = d.layout.rank_stride
        self._stride = S
        lead = (self.R * S,) if self.packed else (self.R, S)
        return DispatchResult(
            recv_x=self._view(d.recv_x, self.dtype, lead + (self.D,)),
            recv_scores=self._view(d.recv_scores, torch.float32, lead),
            recv_src=self._view(d.recv_src, torch.int32, lead),
            layout=self._layout(d.layout))

    # -- calls -------------------------------------------------------------
    def dispatch_layout(self, topk_expert_ids_TK: torch.Tensor, num_tokens_per_rank: int,
                        stream=None, host_counts: bool = False):
        """Layout only. With host_counts=True also returns the per-expert
        counts as a CPU tensor (synchronises; refused while capturing)."""
        host = torch.empty(self.E, dtype=torch.int32) if host_counts else None
        L = ep_dispatch_layout(self.handle, topk_expert_ids_TK, topk_expert_ids_TK.shape[0],
                               num_tokens_per_rank, stream, host)
        lay = self._layout(L)
        return (lay, host) if host_counts else lay

    def dispatch(self, x_TD: torch.Tensor, topk_scores_TK: torch.Tensor,
                 topk_expert_ids_TK: torch.Tensor, num_tokens_per_rank: int | None = None,
                 stream=None) -> DispatchResult:
        _check_dtype(x_TD, self.dtype, "x_TD")
        T = x_TD.shape[0]
        N = T if num_tokens_per_rank is None else num_tokens_per_rank
        d = ep_dispatch(self.handle, x_TD, topk_scores_TK, topk_expert_ids_TK, T, N, stream)
        return self._dispatch_result(d)

    def dispatch_permute(self, x_TD: torch.Tensor, topk_scores_TK: torch.Tensor,
                         stream=None) -> DispatchResult:
        _check_dtype(x_TD, self.dtype, "x_TD")
        return self._dispatch_result(ep_dispatch_permute(self.handle, x_TD, topk_scores_TK,
                                                         stream))

    def combine(self, y_recv: torch.Tensor, topk_scores_TK: torch.Tensor,
                out: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
                stream=None) -> torch.Tensor:
        _check_dtype(y_recv, self.dtype, "y_recv")
        T = topk_scores_TK.shape[0]
        if out is None:
            od = self.dtype if out_dtype is None else out_dtype
            out = torch.empty((T, self.D), dtype=od, device=self.device)
        if out.dtype not in _TORCH_TO_EP:
            raise TypeError(f"out dtype must be bfloat16 or float32, got {out.dtype}")
        ep_combine(self.handle, y_recv, topk_scores_TK, T, out, _TORCH_TO_EP[out.dtype], stream)
        return out

    def combine_backward(self, grad_out: torch.Tensor, y_recv: torch.Tensor | None,
                         topk_scores_TK: torch.Tensor, grad_y: torch.Tensor | None = None,
                         want_scores: bool = True, stream=None):
        """(grad_y [R, S, D], grad_scores [T, K] or None) for the last dispatch.
        grad_y rows that no pair references are left as they were."""
        _check_dtype(grad_out, self.dtype, "grad_out")
        T = topk_scores_TK.shape[0]
        if grad_y is None:
            S = self._last_stride()
            lead = (self.R * S,) if self.packed else (self.R, S)
            grad_y = torch.empty(lead + (self.D,), dtype=self.dtype, device=self.device)
        gs = torch.empty((T, self.K), dtype=torch.float32, device=self.device) \
            if want_scores else None
        ep_combine_backward(self.handle, grad_out, y_recv, topk_scores_TK, T, grad_y, gs, stream)
        return grad_y, gs

    def dispatch_backward(self, grad_recv_x: torch.Tensor, num_tokens: int,
                          grad_recv_scores: torch.Tensor | None = None,
                          out_dtype: torch.dtype | None = None, stream=None):
        """(grad_x [T, D], grad_scores [T, K] or None) for the last dispatch."""
        _check_dtype(grad_recv_x, self.dtype, "grad_recv_x")
        od = self.dtype if out_dtype is None else out_dtype
        gx = torch.empty((num_tokens, self.D), dtype=od, device=self.device)
        gs = None
        if grad_recv_scores is not None:
            gs = torch.empty((num_tokens, self.K), dtype=torch.float32, device=self.device)
        ep_dispatch_backward(self.handle, grad_recv_x, grad_recv_scores, num_tokens, gx,
                             _TORCH_TO_EP[od], gs, stream)
        return gx, gs

    def dispatch_dedup(self, x_TD: torch.Tensor, topk_scores_TK: torch.Tensor,
                       topk_expert_ids_TK: torch.Tensor, num_tokens_per_rank: int | None = None,
                       stream=None) -> DedupResult:
        """One receive row per distinct (token, rank)."""
        _check_dtype(x_TD, self.dtype, "x_TD")
        T = x_TD.shape[0]
        N = T if num_tokens_per_rank is None else num_tokens_per_rank
        d = ep_dispatch_dedup(self.handle, x_TD, topk_scores_TK, topk_expert_ids_TK, T, N, stream)
        P, R, K = d.rows_per_rank_stride, self.R, self.K
        lay = self._layout(d.layout)
        return DedupResult(
            recv_x=self._view(d.recv_x, self.dtype, (R, P, self.D)),
            recv_tok_src=self._view(d.recv_tok_src, torch.int32, (R, P)),
            recv_topk_idx=self._view(d.recv_topk_idx, torch.int32, (R, P, K)),
            recv_topk_w=self._view(d.recv_topk_w, torch.float32, (R, P, K)),
            tok_pos=self._view(d.tok_pos, torch.int32, (T, R)),
            layout=lay)

    def dedup_expand(self, topk_expert_ids_TK: torch.Tensor, y_recv: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
        """The receiver's expansion of the last dedupe dispatch into per-expert rows
        (a tensor shaped like a dispatch's recv_x), ready for combine."""
        S = self._last_stride()
        lead = (self.R * S,) if self.packed else (self.R, S)
        if y_recv is None:
            y_recv = torch.empty(lead + (self.D,), dtype=self.dtype, device=self.device)
        ep_dedup_expand(self.handle, topk_expert_ids_TK, y_recv, stream)
        return y_recv

    def expert_gemm(self, x_recv: torch.Tensor, weights: torch.Tensor,
                    y_recv: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """y = x * W_e^T over each expert's receive rows (weights [E, dout, din]),
        from the counts of the last dispatch on this buffer. Returns y_recv with
        the receive layout's leading shape and dout columns."""
        E, dout, din = weights.shape
        if E != self.E:
            raise ValueError(f"weights must have {self.E} experts, got {E}")
        if x_recv.shape[-1] != din:
            raise ValueError(f"x_recv has {x_recv.shape[-1]} columns, weights expect {din}")
        S = self._last_stride()
        lead = (self.R * S,) if self.packed else (self.R, S)
        if y_recv is None:
            y_recv = torch.empty(lead + (dout,), dtype=torch.bfloat16, device=self.device)
        ep_expert_gemm(self.handle, x_recv, weights, din, dout, y_recv, stream)
        return y_recv

    def _last_stride(self) -> int:
        return self._stride

    def device_error(self, stream=None) -> int:
        return ep_get_device_error(self.handle, stream)

    def info(self) -> dict:
        i = ep_buffer_query(self.handle)
        return {f: getattr(i, f) for f, _ in EpBufferInfo._fields_}

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            ep_buffer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
