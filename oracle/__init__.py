"""CPU oracle for MoE token dispatch and combine (numpy front end over ep_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline use it to check and time against. The product package never imports
it, and it shares no code with the CUDA library.

Arrays are numpy: ids int32 [T, K], scores float32 [T, K], hidden rows float32
[T, D] or bf16 bit patterns uint16 [T, D]. Every function below is a thin
ctypes call into the C source, which cites the passages it follows.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from .build import build_oracle

BF16, F32 = 0, 1
ERR_BAD_ID, ERR_ROW_OOB = 1, 2

_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")


class OracleError(RuntimeError):
    pass


def _kind(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"hidden rows must be uint16 (bf16 bits) or float32, got {a.dtype}")


class Oracle:
    """One loaded build of the oracle (mutant=0 is the real one)."""

    def __init__(self, mutant: int = 0, sanitize: bool = False):
        self.mutant = mutant
        self.lib = C.CDLL(build_oracle(mutant, sanitize=sanitize))
        L = self.lib
        i64, i32 = C.c_int64, C.c_int32
        for name, args in {
            "oracle_ceil_div": [i64, i64],
            "oracle_pad_tokens": [i64],
            "oracle_num_max_tokens_pretrain": [i64, i64, i64, i64],
            "oracle_num_max_tokens_inference": [i64, i64, i64],
            "oracle_rank_stride": [i64, i64],
        }.items():
            f = getattr(L, name)
            f.argtypes, f.restype = args, i64
        L.oracle_bf16_from_f32.argtypes, L.oracle_bf16_from_f32.restype = [C.c_float], C.c_uint16
        L.oracle_f32_from_bf16.argtypes, L.oracle_f32_from_bf16.restype = [C.c_uint16], C.c_float
        L.oracle_bf16_from_f64.argtypes, L.oracle_bf16_from_f64.restype = [C.c_double], C.c_uint16
        u32p = C.POINTER(C.c_uint32)
        L.oracle_routing_map.argtypes = [_i32p, _f32p, i64, i64, i32, i32, _u8p, _f32p, u32p]
        L.oracle_layout.argtypes = [_i32p, i64, i64, i32, i32, i32, i32, _i32p, _i32p, _i32p,
                                    _i32p, _i32p, _i32p, C.POINTER(C.c_int64), u32p]
        L.oracle_dispatch.argtypes = [C.c_void_p, i64, _f32p, _i32p, i64, i64, i32, i32, i32, i32,
                                      C.c_void_p, _f32p, _i32p, _i32p, _i32p, _i32p, _i32p,
                                      _i32p, _i32p, C.POINTER(C.c_int64), u32p]
        L.oracle_combine.argtypes = [C.c_void_p, C.c_int, i64, _f32p, _i32p, _i32p, i64, i64,
                                     i32, i32, i32, C.c_void_p, C.c_int, u32p]
        vp = C.c_void_p
        L.oracle_combine_backward.argtypes = [vp, C.c_int, vp, C.c_int, i64, _f32p, _i32p, _i32p,
                                              i64, i64, i32, i32, i32, vp, vp, u32p]
        L.oracle_dispatch_backward.argtypes = [vp, C.c_int, i64, vp, _i32p, _i32p, i64, i64, i32,
                                               i32, i32, vp, C.c_int, vp, u32p]
        L.oracle_expert_gemm.argtypes = [vp, vp, _i32p, _i32p, i32, i64, i64, vp]
        L.oracle_dispatch_dedup.argtypes = [vp, i64, _f32p, _i32p, i64, i64, i32, i32, i32, vp,
                                            _i32p, _i32p, _f32p, _i32p, _i32p, u32p]
        L.oracle_dedup_expand.argtypes = [vp, i64, _i32p, _i32p, _i32p, i64, i32, i32, i32, vp]
        for name in ("oracle_routing_map", "oracle_layout", "oracle_dispatch", "oracle_combine",
                     "oracle_combine_backward", "oracle_dispatch_backward",
                     "oracle_expert_gemm", "oracle_dispatch_dedup", "oracle_dedup_expand"):
            getattr(L, name).restype = C.c_int

    # -- scalars ------------------------------------------------------------
    def ceil_div(self, a: int, b: int) -> int:
        return int(self.lib.oracle_ceil_div(a, b))

    def pad_tokens(self, n: int) -> int:
        return int(self.lib.oracle_pad_tokens(n))

    def num_max_tokens_pretrain(self, local_batch_size, seq_len, cp, tp) -> int:
        return int(self.lib.oracle_num_max_tokens_pretrain(local_batch_size, seq_len, cp, tp))

    def num_max_tokens_inference(self, max_num_batched_tokens, cp, tp) -> int:
        return int(self.lib.oracle_num_max_tokens_inference(max_num_batched_tokens, cp, tp))

    def rank_stride(self, N: int, K: int) -> int:
        return int(self.lib.oracle_rank_stride(N, K))

    def bf16_from_f32(self, a) -> np.ndarray:
        a = np.asarray(a, dtype=np.float32).ravel()
        return np.array([self.lib.oracle_bf16_from_f32(float(v)) for v in a], dtype=np.uint16)

    def bf16_from_f64(self, a) -> np.ndarray:
        a = np.asarray(a, dtype=np.float64).ravel()
        return np.array([self.lib.oracle_bf16_from_f64(float(v)) for v in a], dtype=np.uint16)

    def f32_from_bf16(self, h) -> np.ndarray:
        h = np.asarray(h, dtype=np.uint16).ravel()
        return np.array([self.lib.oracle_f32_from_bf16(int(v)) for v in h], dtype=np.float32)

    # -- arrays -------------------------------------------------------------
    def routing_map(self, ids, scores, N: int, E: int):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        T, K = ids.shape
        P = self.pad_tokens(N)
        m = np.zeros((P, E), dtype=np.uint8)
        pr = np.zeros((P, E), dtype=np.float32)
        err = C.c_uint32(0)
        rc = self.lib.oracle_routing_map(ids.ravel(), scores.ravel(), T, N, K, E, m.ravel(),
                                         pr.ravel(), C.byref(err))
        if rc:
            raise OracleError(f"oracle_routing_map rc={rc}")
        return m.astype(bool), pr, int(err.value)

    def layout(self, ids, N: int, E: int, R: int, packed: bool = False) -> dict:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, K = ids.shape
        out = {
            "cnt": np.zeros(E, np.int32), "expert_offset": np.zeros(E, np.int32),
            "rows_per_rank": np.zeros(R, np.int32), "rank_prefix": np.zeros(R, np.int32),
            "tokens_in_rank": np.zeros(R, np.int32), "pos": np.zeros((T, K), np.int32),
        }
        S = C.c_int64(0)
        err = C.c_uint32(0)
        rc = self.lib.oracle_layout(ids.ravel() if T else np.zeros(1, np.int32), T, N, K, E, R,
                                    int(packed), out["cnt"], out["expert_offset"], out["rows_per_rank"],
                                    out["rank_prefix"], out["tokens_in_rank"],
                                    out["pos"].ravel() if T else np.zeros(1, np.int32),
                                    C.byref(S), C.byref(err))
        if rc:
            raise OracleError(f"oracle_layout rc={rc}")
        out["S"] = int(S.value)
        out["err"] = int(err.value)
        return out

    def dispatch(self, x, scores, ids, N: int, E: int, R: int, fill: int = 0,
                 packed: bool = False) -> dict:
        """Layout plus permute. Receive buffers hold R*S rows; rows that no pair
        lands on keep the byte ``fill``."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        x = np.ascontiguousarray(x)
        _kind(x)
        T, K = ids.shape
        D = x.shape[1]
        row_bytes = D * x.itemsize
        S = self.rank_stride(N, K)
        rows = R * S
        recv_x = np.full((rows, D), 0, dtype=x.dtype)
        recv_x.view(np.uint8)[...] = fill
        recv_scores = np.zeros(rows, np.float32)
        recv_src = np.full(rows, -1, np.int32)
        lay = {
            "cnt": np.zeros(E, np.int32), "expert_offset": np.zeros(E, np.int32),
            "rows_per_rank": np.zeros(R, np.int32), "rank_prefix": np.zeros(R, np.int32),
            "tokens_in_rank": np.zeros(R, np.int32), "pos": np.zeros((T, K), np.int32),
        }
        Sv = C.c_int64(0)
        err = C.c_uint32(0)
        one_i = np.zeros(1, np.int32)
        rc = self.lib.oracle_dispatch(
            x.ctypes.data if T else None, row_bytes, scores.ravel() if T else np.zeros(1, np.float32),
            ids.ravel() if T else one_i, T, N, K, E, R, int(packed),
            recv_x.ctypes.data if rows else None,
            recv_scores if rows else np.zeros(1, np.float32), recv_src if rows else one_i,
            lay["cnt"], lay["expert_offset"], lay["rows_per_rank"], lay["rank_prefix"],
            lay["tokens_in_rank"], lay["pos"].ravel() if T else one_i, C.byref(Sv), C.byref(err))
        if rc:
            raise OracleError(f"oracle_dispatch rc={rc}")
        lay.update(S=int(Sv.value), err=int(err.value), recv_x=recv_x, recv_scores=recv_scores,
                   recv_src=recv_src, packed=bool(packed))
        return lay

    def combine(self, y, scores, pos, rank_prefix, S: int, R: int, out_dtype: str = "same",
                packed: bool = False):
        """out[T, D]; out_dtype "same" (y's kind), "bf16" or "f32". Returns (out, err)."""
        y = np.ascontiguousarray(y)
        yk = _kind(y)
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        rank_prefix = np.ascontiguousarray(rank_prefix, dtype=np.int32)
        T, K = pos.shape
        D = y.shape[1]
        ok = {"same": yk, "bf16": BF16, "f32": F32}[out_dtype]
        out = np.zeros((T, D), dtype=np.uint16 if ok == BF16 else np.float32)
        err = C.c_uint32(0)
        rc = self.lib.oracle_combine(y.ctypes.data if y.size else None, yk, D,
                                     scores.ravel() if T else np.zeros(1, np.float32),
                                     pos.ravel() if T else np.zeros(1, np.int32), rank_prefix,
                                     S, T, K, R, int(packed), out.ctypes.data if T else None, ok,
                                     C.byref(err))
        if rc:
            raise OracleError(f"oracle_combine rc={rc}")
        return out, int(err.value)


    # -- backward ------------------------------------------------------------
    def combine_backward(self, grad_out, y, scores, pos, rank_prefix, S: int, R: int,
                         grad_y_fill: int = 0, packed: bool = False):
        """(grad_y [R*S, D] of y's kind, grad_scores [T, K] fp32, err). Rows of
        grad_y that no valid pair references keep the byte grad_y_fill."""
        grad_out = np.ascontiguousarray(grad_out)
        y = np.ascontiguousarray(y)
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        rank_prefix = np.ascontiguousarray(rank_prefix, dtype=np.int32)
        T, K = pos.shape
        D = y.shape[1]
        grad_y = np.zeros_like(y)
        grad_y.view(np.uint8)[...] = grad_y_fill
        gs = np.zeros((T, K), np.float32)
        err = C.c_uint32(0)
        rc = self.lib.oracle_combine_backward(
            grad_out.ctypes.data if T else None, _kind(grad_out), y.ctypes.data if y.size else None,
            _kind(y), D, scores.ravel() if T else np.zeros(1, np.float32),
            pos.ravel() if T else np.zeros(1, np.int32), rank_prefix, S, T, K, R, int(packed),
            grad_y.ctypes.data if grad_y.size else None, gs.ctypes.data if T else None,
            C.byref(err))
        if rc:
            raise OracleError(f"oracle_combine_backward rc={rc}")
        return grad_y, gs, int(err.value)

    def dispatch_backward(self, grad_recv, grad_recv_scores, pos, rank_prefix, S: int, R: int,
                          out_dtype: str = "same", packed: bool = False):
        """(grad_x [T, D], grad_scores [T, K] fp32 or None, err)."""
        grad_recv = np.ascontiguousarray(grad_recv)
        gk = _kind(grad_recv)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        rank_prefix = np.ascontiguousarray(rank_prefix, dtype=np.int32)
        T, K = pos.shape
        D = grad_recv.shape[1]
        ok = {"same": gk, "bf16": BF16, "f32": F32}[out_dtype]
        gx = np.zeros((T, D), dtype=np.uint16 if ok == BF16 else np.float32)
        grs = None if grad_recv_scores is None else np.ascontiguousarray(grad_recv_scores,
                                                                          dtype=np.float32)
        gs = None if grs is None else np.zeros((T, K), np.float32)
        err = C.c_uint32(0)
        rc = self.lib.oracle_dispatch_backward(
            grad_recv.ctypes.data if grad_recv.size else None, gk, D,
            None if grs is None else grs.ctypes.data, pos.ravel() if T else np.zeros(1, np.int32),
            rank_prefix, S, T, K, R, int(packed), gx.ctypes.data if T else None, ok,
            None if gs is None or not T else gs.ctypes.data, C.byref(err))
        if rc:
            raise OracleError(f"oracle_dispatch_backward rc={rc}")
        return gx, gs, int(err.value)


    # -- expert consumer -----------------------------------------------------
    def expert_gemm(self, x, w, cnt, expert_offset, fill: int = 0):
        """y [rows, dout] bf16 bits: each expert's rows times its weight
        matrix transposed (fp64 sum, one rounding); other rows keep `fill`."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        w = np.ascontiguousarray(w, dtype=np.uint16)
        cnt = np.ascontiguousarray(cnt, dtype=np.int32)
        off = np.ascontiguousarray(expert_offset, dtype=np.int32)
        E, dout, din = w.shape
        y = np.full((x.shape[0], dout), fill, dtype=np.uint16)
        rc = self.lib.oracle_expert_gemm(x.ctypes.data, w.ctypes.data, cnt, off, E, din, dout,
                                         y.ctypes.data)
        if rc:
            raise OracleError(f"oracle_expert_gemm rc={rc}")
        return y


    # -- per-rank dedupe --------------------------------------------------------
    def dispatch_dedup(self, x, scores, ids, N: int, E: int, R: int, fill: int = 0) -> dict:
        """One receive row per (token, rank): recv_tok_x [R*P, D], recv_tok_src
        [R*P], recv_topk_idx [R*P, K], recv_topk_w [R*P, K], tok_pos [T, R],
        tokens_in_rank [R]; rows past each rank's total keep `fill`."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        x = np.ascontiguousarray(x)
        _kind(x)
        T, K = ids.shape
        D = x.shape[1]
        rows = R * self.pad_tokens(N)
        rx = np.zeros((max(rows, 1), D), dtype=x.dtype)
        rx.view(np.uint8)[...] = fill
        src = np.full(max(rows, 1), -1, np.int32)
        idx = np.full((max(rows, 1), K), -2, np.int32)
        wts = np.zeros((max(rows, 1), K), np.float32)
        tpos = np.zeros((max(T, 1), R), np.int32)
        tir = np.zeros(R, np.int32)
        err = C.c_uint32(0)
        rc = self.lib.oracle_dispatch_dedup(
            x.ctypes.data if T else None, D * x.itemsize,
            scores.ravel() if T else np.zeros(1, np.float32),
            ids.ravel() if T else np.zeros(1, np.int32), T, N, K, E, R, rx.ctypes.data,
            src, idx.ravel(), wts.ravel(), tpos.ravel(), tir, C.byref(err))
        if rc:
            raise OracleError(f"oracle_dispatch_dedup rc={rc}")
        return {"recv_tok_x": rx[:rows], "recv_tok_src": src[:rows], "recv_topk_idx": idx[:rows],
                "recv_topk_w": wts[:rows], "tok_pos": tpos[:T], "tokens_in_rank": tir,
                "P": self.pad_tokens(N), "err": int(err.value)}

    def dedup_expand(self, recv_tok_x, tok_pos, pos, ids, E: int, R: int, rows: int,
                     fill: int = 0):
        """Expert-layout rows y [rows, D] from the dedupe rows."""
        recv_tok_x = np.ascontiguousarray(recv_tok_x)
        tok_pos = np.ascontiguousarray(tok_pos, dtype=np.int32)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, K = ids.shape
        D = recv_tok_x.shape[1]
        y = np.zeros((rows, D), dtype=recv_tok_x.dtype)
        y.view(np.uint8)[...] = fill
        rc = self.lib.oracle_dedup_expand(recv_tok_x.ctypes.data, D * recv_tok_x.itemsize,
                                          tok_pos.ravel() if T else np.zeros(1, np.int32),
                                          pos.ravel() if T else np.zeros(1, np.int32),
                                          ids.ravel() if T else np.zeros(1, np.int32), T, K, E,
                                          R, y.ctypes.data)
        if rc:
            raise OracleError(f"oracle_dedup_expand rc={rc}")
        return y


_default: Oracle | None = None


def get() -> Oracle:
    """The real oracle (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default
