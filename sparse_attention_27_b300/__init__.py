"""Python binding of libsa27 (hybrid compressed attention, CSA + HCA, on B300).

Argument marshalling only: every function below has the name of the C entry
point it calls (declared in ``include/sa.h``), passes device pointers of
torch tensors (``data_ptr()``), sizes and the current CUDA stream, and turns
a non-zero status into ``SaError``.  All computation happens in the library's
CUDA kernels; there is no other implementation behind these names.  If the
library is missing, importing this package raises: there is no fallback.

Build the library with ``python -m sparse_attention_27_b300.build``.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsa27.so")

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CUDA = 0, 1, 2, 3
SA_ERR_DEVICE_TIMEOUT, SA_ERR_BOUNDS, SA_ERR_NAN = 4, 5, 6
SA_F32, SA_BF16, SA_MXFP4 = 0, 1, 2

EXPORTS = (
    "sa_status_string", "csa_compress", "csa_index_topk", "csa_index_topk_workspace_bytes",
    "csa_attend", "csa_attend_workspace_bytes", "hca_compress_attend",
    "hca_compress_attend_workspace_bytes", "attn_merge", "csa_index_topk_noalloc",
    "sa_mxfp4_quantize", "csa_decode", "csa_attend_backward", "hca_attend_backward",
    "sa_compress_backward", "sa_decode_step", "sa_decode_step_workspace_bytes", "sa_ring_write",
    "sa_compress_channels",
)


class SaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libsa27.so not built at {LIB_PATH}; run python -m sparse_attention_27_b300.build")

_lib = C.CDLL(LIB_PATH)
_vp, _i, _i64, _f, _sz = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_size_t

_lib.sa_status_string.argtypes = [_i]
_lib.sa_status_string.restype = C.c_char_p
_lib.csa_compress.argtypes = [_i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp,
                              _vp, _vp, _vp, _i, _vp, _vp]
_lib.csa_index_topk.argtypes = [_i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp,
                                _vp, _vp, _vp, _vp, _sz, _vp, _vp]
_lib.csa_index_topk_workspace_bytes.argtypes = [_i, _i, _i, _i]
_lib.csa_index_topk_workspace_bytes.restype = _sz
_lib.csa_index_topk_noalloc.argtypes = [_i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i,
                                        _vp, _vp, _vp, _vp]
_lib.sa_mxfp4_quantize.argtypes = [_vp, _i64, _vp, _vp, _vp]
_lib.csa_attend_backward.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _i,
                                     _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _vp]
_lib.hca_attend_backward.argtypes = [_i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _i, _vp,
                                     _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.sa_compress_backward.argtypes = [_i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp,
                                      _i, _vp, _vp, _vp, _vp, _vp]
_lib.csa_decode.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                            _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp,
                            _vp]
_lib.sa_decode_step.argtypes = ([_i] * 9 + [_f] + [_vp] * 12 + [_i] + [_vp] * 2 + [_i] +
                                 [_vp] * 2 + [_i] + [_vp] * 3 + [_i] + [_vp] * 2 + [_i] +
                                 [_vp, _i] + [_vp] * 5 + [_sz, _vp, _vp])
_lib.sa_decode_step_workspace_bytes.argtypes = [_i] * 6
_lib.sa_ring_write.argtypes = [_i, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp]
_lib.sa_compress_channels.argtypes = [_i, _i, _i, _i, _vp, _vp, _i, _vp, _vp, _i, _vp, _i, _vp,
                                      _vp]
_lib.sa_decode_step_workspace_bytes.restype = _sz
_lib.csa_attend.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _i, _vp, _vp,
                            _vp, _i, _vp, _i, _vp, _vp, _sz, _vp, _vp]
_lib.csa_attend_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
_lib.csa_attend_workspace_bytes.restype = _sz
_lib.hca_compress_attend.argtypes = [_i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _i,
                                     _vp, _vp, _i, _vp, _vp, _i, _vp, _i, _vp, _vp, _sz, _vp, _vp]
_lib.hca_compress_attend_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
_lib.hca_compress_attend_workspace_bytes.restype = _sz
_lib.attn_merge.argtypes = [_i, _vp, _vp, _i64, _i, _vp, _i, _vp, _vp, _vp]


def library() -> C.CDLL:
    return _lib


def status_string(s: int) -> str:
    return _lib.sa_status_string(int(s)).decode()


def _p(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(s: int, where: str) -> None:
    if s != SA_OK:
        raise SaError(s, where)


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SA_F32
    if t.dtype == torch.bfloat16:
        return SA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def csa_compress(dtype, ik_dtype, B, d, dI, m, k_raw, v_raw, ik_raw, z, R, blk_lo, blk_hi,
                 max_blocks, k_c, v_c, ik_c, ik_c_scales, N_cap, err=None, stream=None):
    _check(_lib.csa_compress(dtype, ik_dtype, B, d, dI, m, _p(k_raw), _p(v_raw), _p(ik_raw), _p(z),
                             R, _p(blk_lo), _p(blk_hi), max_blocks, _p(k_c), _p(v_c), _p(ik_c),
                             _p(ik_c_scales), N_cap, _p(err), _stream(stream)), "csa_compress")


def csa_index_topk_workspace_bytes(B, T, N_cap, k) -> int:
    return int(_lib.csa_index_topk_workspace_bytes(B, T, N_cap, k))


def csa_index_topk(q_dtype, B, T, HI, dI, m, k, q_idx, q_scales, w, ik_c, ik_scales, N_cap, q_pos,
                   idx, scores_out=None, scores_in=None, ws=None, ws_bytes=0, err=None,
                   stream=None):
    _check(_lib.csa_index_topk(q_dtype, B, T, HI, dI, m, k, _p(q_idx), _p(q_scales), _p(w),
                               _p(ik_c), _p(ik_scales), N_cap, _p(q_pos), _p(idx),
                               _p(scores_out), _p(scores_in), _p(ws), ws_bytes, _p(err),
                               _stream(stream)), "csa_index_topk")


def csa_index_topk_noalloc(q_dtype, B, T, HI, dI, m, k, q_idx, q_scales, w, ik_c, ik_scales,
                           N_cap, q_pos, idx, err=None, stream=None):
    """csa_index_topk without a workspace: the scores live in the library's
    own fixed device array (at most SA_NOALLOC_MAX_SCORES = B*T*N_cap)."""
    _check(_lib.csa_index_topk_noalloc(q_dtype, B, T, HI, dI, m, k, _p(q_idx), _p(q_scales), _p(w),
                                       _p(ik_c), _p(ik_scales), N_cap, _p(q_pos), _p(idx), _p(err),
                                       _stream(stream)), "csa_index_topk_noalloc")


NOALLOC_MAX_SCORES = 2097152


def csa_attend_workspace_bytes(dtype, B, T, H, d, k, W) -> int:
    return int(_lib.csa_attend_workspace_bytes(dtype, B, T, H, d, k, W))


def _out_code(o) -> int:
    """dtype code of an output tensor (f32 for anything that is not a tensor)."""
    return dtype_code(o) if isinstance(o, torch.Tensor) else SA_F32


def csa_attend(dtype, B, T, H, d, m, k, W, sm_scale, q, q_pos, k_c, v_c, N_cap, idx, k_raw, v_raw,
               R, o, lse, ws=None, ws_bytes=0, err=None, stream=None):
    """o: f32 or bf16 tensor [B,T,H,d] (its dtype selects the output type)."""
    _check(_lib.csa_attend(dtype, B, T, H, d, m, k, W, sm_scale, _p(q), _p(q_pos), _p(k_c),
                           _p(v_c), N_cap, _p(idx), _p(k_raw), _p(v_raw), R, _p(o), _out_code(o),
                           _p(lse), _p(ws), ws_bytes, _p(err), _stream(stream)), "csa_attend")


def hca_compress_attend_workspace_bytes(dtype, B, T, H, d, N2_cap, W) -> int:
    return int(_lib.hca_compress_attend_workspace_bytes(dtype, B, T, H, d, N2_cap, W))


def hca_compress_attend(dtype, B, T, H, d, m2, W, sm_scale, q, q_pos, k_raw, v_raw, z_hca, R,
                        blk_lo, blk_hi, max_blocks, hk_c, hv_c, N2_cap, o, lse, ws=None,
                        ws_bytes=0, err=None, stream=None):
    _check(_lib.hca_compress_attend(dtype, B, T, H, d, m2, W, sm_scale, _p(q), _p(q_pos),
                                    _p(k_raw), _p(v_raw), _p(z_hca), R, _p(blk_lo), _p(blk_hi),
                                    max_blocks, _p(hk_c), _p(hv_c), N2_cap, _p(o), _out_code(o),
                                    _p(lse), _p(ws), ws_bytes, _p(err), _stream(stream)),
           "hca_compress_attend")


def csa_decode(B, H, d, HI, dI, m, k, W, sm_scale, q, q_idx, w, q_pos, k_raw, v_raw, ik_raw, z,
               R, blk_lo, blk_hi, max_blocks, k_c, v_c, ik_c, N_cap, idx, o, lse, err=None,
               stream=None):
    """The fused CSA layer of one decode step; o: f32 or bf16 tensor [B,H,d]
    (its dtype selects the output type)."""
    _check(_lib.csa_decode(B, H, d, HI, dI, m, k, W, sm_scale, _p(q), _p(q_idx), _p(w),
                           _p(q_pos), _p(k_raw), _p(v_raw), _p(ik_raw), _p(z), R, _p(blk_lo),
                           _p(blk_hi), max_blocks, _p(k_c), _p(v_c), _p(ik_c), N_cap, _p(idx),
                           _p(o), _out_code(o), _p(lse), _p(err), _stream(stream)), "csa_decode")


def sa_compress_channels(dtype, B, d, m, x_raw, z, R, blk_lo, blk_hi, max_blocks, x_c, N_cap,
                         err=None, stream=None):
    """Per-channel softmax pooling of one array: z [B,R,d] f32 logits."""
    _check(_lib.sa_compress_channels(dtype, B, d, m, _p(x_raw), _p(z), R, _p(blk_lo), _p(blk_hi),
                                     max_blocks, _p(x_c), N_cap, _p(err), _stream(stream)),
           "sa_compress_channels")


def sa_ring_write(B, R, pos, rings, rows, err=None, stream=None):
    """Each sequence's new token into the rings: rings[i][b, pos[b] % R] =
    rows[i][b] for every pair (ring [B,R,...], rows [B,...], same dtype)."""
    n = len(rings)
    if n != len(rows) or not 1 <= n <= 8:
        raise SaError(SA_ERR_INVALID_ARG, "sa_ring_write")
    ring_p = (C.c_void_p * n)(*[_p(t) for t in rings])
    row_p = (C.c_void_p * n)(*[_p(t) for t in rows])
    nbytes = (C.c_int * n)(*[t[0].numel() * t.element_size() if t.dim() > 1 else t.element_size()
                             for t in rows])
    _check(_lib.sa_ring_write(B, R, _p(pos), n, ring_p, row_p, nbytes, _p(err), _stream(stream)),
           "sa_ring_write")


def sa_decode_step_workspace_bytes(B, H, N_cap, k, W, N2_cap) -> int:
    """Workspace bytes of sa_decode_step (0: the shape is not taken)."""
    return int(_lib.sa_decode_step_workspace_bytes(B, H, N_cap, k, W, N2_cap))


def sa_decode_step(B, H, d, HI, dI, m, k, W, m2, sm_scale, q, q_idx, w, q_hca, q_pos, k_raw,
                   v_raw, ik_raw, z, hk_raw, hv_raw, hz, R, blk_lo, blk_hi, max_blocks, hblk_lo,
                   hblk_hi, max_blocks2, k_c, v_c, ik_c, N_cap, hk_c, hv_c, N2_cap, idx, o, lse,
                   ho, hlse, ws, ws_bytes=None, err=None, stream=None):
    """Both layers of one decode step in one launch; o and ho: f32 or bf16
    tensors [B,H,d] of the same dtype (it selects the output type)."""
    if _out_code(o) != _out_code(ho):
        raise SaError(SA_ERR_INVALID_ARG, "sa_decode_step")
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(_lib.sa_decode_step(B, H, d, HI, dI, m, k, W, m2, sm_scale, _p(q), _p(q_idx), _p(w),
                               _p(q_hca), _p(q_pos), _p(k_raw), _p(v_raw), _p(ik_raw), _p(z),
                               _p(hk_raw), _p(hv_raw), _p(hz), R, _p(blk_lo), _p(blk_hi),
                               max_blocks, _p(hblk_lo), _p(hblk_hi), max_blocks2, _p(k_c),
                               _p(v_c), _p(ik_c), N_cap, _p(hk_c), _p(hv_c), N2_cap, _p(idx),
                               _out_code(o), _p(o), _p(lse), _p(ho), _p(hlse), _p(ws), ws_bytes,
                               _p(err), _stream(stream)), "sa_decode_step")


def csa_attend_backward(dtype, B, T, H, d, m, k, W, sm_scale, q, q_pos, k_c, v_c, N_cap, idx,
                        k_raw, v_raw, R, o, lse, dout, dq, dk_c, dv_c, dk_raw, dv_raw, err=None,
                        stream=None):
    """Gradient of csa_attend for the given selection; adds into the f32
    gradient tensors dq, dk_c, dv_c, dk_raw, dv_raw."""
    _check(_lib.csa_attend_backward(dtype, B, T, H, d, m, k, W, sm_scale, _p(q), _p(q_pos),
                                    _p(k_c), _p(v_c), N_cap, _p(idx), _p(k_raw), _p(v_raw), R,
                                    _p(o), _p(lse), _p(dout), _p(dq), _p(dk_c), _p(dv_c),
                                    _p(dk_raw), _p(dv_raw), _p(err), _stream(stream)),
           "csa_attend_backward")


def hca_attend_backward(dtype, B, T, H, d, m2, W, sm_scale, q, q_pos, hk_c, hv_c, N2_cap, k_raw,
                        v_raw, R, o, lse, dout, dq, dhk_c, dhv_c, dk_raw, dv_raw, err=None,
                        stream=None):
    """Gradient of the HCA attention (all visible HCA rows and the window)."""
    _check(_lib.hca_attend_backward(dtype, B, T, H, d, m2, W, sm_scale, _p(q), _p(q_pos),
                                    _p(hk_c), _p(hv_c), N2_cap, _p(k_raw), _p(v_raw), R, _p(o),
                                    _p(lse), _p(dout), _p(dq), _p(dhk_c), _p(dhv_c), _p(dk_raw),
                                    _p(dv_raw), _p(err), _stream(stream)), "hca_attend_backward")


def sa_compress_backward(dtype, B, d, m, k_raw, v_raw, z, R, blk_lo, blk_hi, max_blocks, dk_c,
                         dv_c, N_cap, dk_raw, dv_raw, dz, err=None, stream=None):
    """Gradient of the K/V pooling of blocks [blk_lo, blk_hi); adds into
    dk_raw, dv_raw and dz."""
    _check(_lib.sa_compress_backward(dtype, B, d, m, _p(k_raw), _p(v_raw), _p(z), R, _p(blk_lo),
                                     _p(blk_hi), max_blocks, _p(dk_c), _p(dv_c), N_cap,
                                     _p(dk_raw), _p(dv_raw), _p(dz), _p(err), _stream(stream)),
           "sa_compress_backward")


def sa_mxfp4_quantize(x, codes, scales, stream=None):
    """x: bf16 tensor whose element count is a multiple of 32; codes: uint8
    with half as many elements; scales: uint8 with one per 32 elements."""
    nblk = x.numel() // 32
    _check(_lib.sa_mxfp4_quantize(_p(x), nblk, _p(codes), _p(scales), _stream(stream)),
           "sa_mxfp4_quantize")


def attn_merge(o_parts, lse_parts, o, lse, err=None, stream=None):
    """o_parts: list of [rows, d] f32 tensors; lse_parts: list of [rows] f32."""
    n = len(o_parts)
    rows, d = o_parts[0].shape[0], o_parts[0].shape[-1]
    op = (C.c_void_p * n)(*[t.data_ptr() for t in o_parts])
    lp = (C.c_void_p * n)(*[t.data_ptr() for t in lse_parts])
    _check(_lib.attn_merge(n, C.cast(op, C.c_void_p), C.cast(lp, C.c_void_p), rows, d, _p(o),
                           dtype_code(o), _p(lse), _p(err), _stream(stream)), "attn_merge")
