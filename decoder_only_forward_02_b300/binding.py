"""ctypes binding of the C ABI in ``include/nc.h``.

Argument marshalling only: every step of the forward pass runs in the CUDA kernels of
``libnc.so``.  PyTorch supplies device memory and streams.  There is no fallback: if the
library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnc.so")

NC_OK = 0
STATUS_NAMES = {0: "NC_OK", 1: "NC_ERR_INVALID_ARG", 2: "NC_ERR_UNSUPPORTED", 3: "NC_ERR_WORKSPACE",
                4: "NC_ERR_CUDA", 5: "NC_ERR_DEVICE_TIMEOUT", 6: "NC_ERR_TOKEN_RANGE"}
KERNEL_CLASSES = ["embed_smear", "qkv_rope_qknorm_ve", "attention", "oproj_residual", "fc_relu2",
                  "proj_residual", "lmhead_softcap", "cross_entropy", "lmhead_grad", "mlp_grad", "oproj_grad",
                  "rmsnorm_grad", "fp8_quantize"]
SS_GROUP = 128   # columns per partial sum of squares
QKV_GATE_ROWS = 16   # rows after each kv head's v rows in a value-embedding layer's packed q|k|v weight

c_int_p = ctypes.POINTER(ctypes.c_int)
c_void_pp = ctypes.POINTER(ctypes.c_void_p)


class NcConfig(ctypes.Structure):
    _fields_ = [
        ("n_layer", ctypes.c_int), ("n_embd", ctypes.c_int), ("n_head", ctypes.c_int),
        ("n_kv_head", ctypes.c_int), ("head_dim", ctypes.c_int), ("mlp_hidden", ctypes.c_int),
        ("vocab_size", ctypes.c_int), ("seq_len_ctx", ctypes.c_int),
        ("window_left", c_int_p), ("has_ve", ctypes.POINTER(ctypes.c_ubyte)),
        ("use_smear", ctypes.c_int), ("use_backout", ctypes.c_int), ("embed_norm", ctypes.c_int),
        ("smear_gate_channels", ctypes.c_int), ("ve_gate_channels", ctypes.c_int),
        ("ve_gate_scale", ctypes.c_float), ("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float),
        ("softcap", ctypes.c_float), ("logits_bf16", ctypes.c_int), ("fp8", ctypes.c_int),
    ]


class NcWeights(ctypes.Structure):
    _fields_ = [
        ("wte", ctypes.c_void_p), ("wq", c_void_pp), ("wk", c_void_pp), ("wv", c_void_pp),
        ("wo", c_void_pp), ("wfc", c_void_pp), ("wproj", c_void_pp), ("ve_table", c_void_pp),
        ("ve_gate", c_void_pp), ("smear_gate", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
        ("resid_lambdas", ctypes.POINTER(ctypes.c_float)), ("x0_lambdas", ctypes.POINTER(ctypes.c_float)),
        ("backout_lambda", ctypes.c_float),
    ]


_SIGS = {
    "nc_model_packed_bytes": (ctypes.c_int, [ctypes.POINTER(NcConfig), ctypes.POINTER(ctypes.c_size_t)]),
    "nc_model_create": (ctypes.c_int, [ctypes.POINTER(NcConfig), ctypes.POINTER(NcWeights), ctypes.c_void_p,
                                       ctypes.c_size_t, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    "nc_workspace_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_size_t)]),
    "nc_workspace_bytes_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_size_t)]),
    "nc_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "nc_forward_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "nc_forward_static_scratch": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_void_p, ctypes.c_void_p]),
    "nc_get_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "nc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "nc_last_cuda_error": (ctypes.c_char_p, []),
    "nc_model_destroy": (None, [ctypes.c_void_p]),
    "nc_timing_enable": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "nc_timing_read": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_int)]),
    "nc_kernel_class_name": (ctypes.c_char_p, [ctypes.c_int]),
    "nc_forward_launch_count": (ctypes.c_int, [ctypes.c_void_p]),
    "nc_forward_loss_launch_count": (ctypes.c_int, [ctypes.c_void_p]),
    "nc_kv_launch_count": (ctypes.c_int, [ctypes.c_void_p]),
    "nc_kv_cache_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "nc_workspace_bytes_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "nc_prefill": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                  ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                  ctypes.c_void_p]),
    "nc_decode_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "nc_workspace_bytes_loss": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_size_t)]),
    "nc_forward_loss": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
                        + [ctypes.c_void_p] * 4 + [ctypes.c_size_t, ctypes.c_void_p]),
    "nc_workspace_bytes_grad_tail": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                    ctypes.POINTER(ctypes.c_size_t)]),
    "nc_forward_loss_grad_tail": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                                 ctypes.c_int] + [ctypes.c_void_p] * 7 + [ctypes.c_size_t,
                                                                                         ctypes.c_void_p]),
    "nc_grad_tail_launch_count": (ctypes.c_int, [ctypes.c_void_p]),
    # per-kernel entry points (include/nc_ops.h)
    "nc_op_gemm": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]),
    "nc_op_gemm_residual": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_float]
                            + [ctypes.c_void_p] * 7),
    "nc_op_qkv": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 6 +
                  [ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5),
    "nc_op_rope_table": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                        ctypes.c_void_p]),
    "nc_op_attention": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int] * 6 +
                        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "nc_op_embed_smear": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_float, ctypes.c_float] + [ctypes.c_void_p] * 6),
    "nc_op_lmhead_ce": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_float, ctypes.c_float] + [ctypes.c_void_p] * 5),
    "nc_op_ce_scratch_bytes": (ctypes.c_size_t, [ctypes.c_int]),
    "nc_op_test_wait_timeout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 3 +
                                [ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong, ctypes.c_int, ctypes.c_void_p,
                                 ctypes.c_void_p]),
    "nc_op_ce_finalize": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_int] + [ctypes.c_void_p] * 4 + [ctypes.c_size_t] +
                          [ctypes.c_void_p] * 4),
    "nc_op_gemm_t": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 6 +
                     [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                      ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "nc_op_gemm_split_ws_bytes": (ctypes.c_size_t, [ctypes.c_int] * 4),
    "nc_op_fp8_scratch_bytes": (ctypes.c_size_t, []),
    "nc_op_fp8_quantize": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_float] + [ctypes.c_void_p] * 4),
    "nc_op_gemm_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 4 +
                       [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                        ctypes.c_void_p, ctypes.c_void_p]),
    "nc_op_lmhead_ce_grad": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_float] +
                             [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "nc_op_mlp_hidden_grad": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_float] + [ctypes.c_void_p] * 4),
    "nc_op_rms_backward": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_int, ctypes.c_float] +
                           [ctypes.c_void_p] * 3),
}

EPI = {"bf16": 0, "relu2_bf16": 2, "softcap_f32": 3, "softcap_bf16": 6, "f32": 7}


class ops:
    """Per-kernel entry points; tensors are CUDA tensors, launches go on the current stream."""

    @staticmethod
    def gemm(A, B, epi="bf16", out=None, ssp=None, C=0, eps=1e-6, cap=15.0, status=None):
        M, K = A.shape
        N = B.shape[0]
        if out is None:
            dt = torch.bfloat16 if epi in ("bf16", "relu2_bf16", "softcap_bf16") else torch.float32
            out = torch.empty((M, N), dtype=dt, device=A.device)
        check(lib().nc_op_gemm(A.data_ptr(), B.data_ptr(), M, N, K, EPI[epi], out.data_ptr(), out.shape[1],
                               _ptr(ssp), C, eps, cap, _ptr(status), _stream_handle(None)), "nc_op_gemm")
        return out

    @staticmethod
    def gemm_t(A, B, a_mn=False, b_mn=False, epi="f32", out=None, ssp=None, C=0, eps=1e-6, cap=15.0, status=None,
               split=False):
        """nc_op_gemm_t: A is [M, K] (a_mn False) or stored [K, M] (a_mn True); B is [N, K] or stored
        [K, N]; returns epi(A . B^T) [M, N].  split: give the call a K-split workspace (fp32 output)."""
        K, M = A.shape if a_mn else A.shape[::-1]
        KB, N = B.shape if b_mn else B.shape[::-1]
        if KB != K:
            raise ValueError("A and B disagree on K")
        if out is None:
            dt = torch.bfloat16 if epi in ("bf16", "relu2_bf16", "softcap_bf16") else torch.float32
            out = torch.empty((M, N), dtype=dt, device=A.device)
        ws, nws = None, 0
        if split:
            nws = lib().nc_op_gemm_split_ws_bytes(M, N, K, out.shape[1])
            ws = torch.empty((max(nws, 16) // 4,), dtype=torch.float32, device=A.device)
        check(lib().nc_op_gemm_t(A.data_ptr(), B.data_ptr(), M, N, K, int(a_mn), int(b_mn), EPI[epi], out.data_ptr(),
                                 out.shape[1], _ptr(ssp), C, eps, cap, _ptr(ws), nws, _ptr(status),
                                 _stream_handle(None)), "nc_op_gemm_t")
        return out

    @staticmethod
    def fp8_quantize(src, ssp=None, eps=1e-6):
        """e4m3 codes (torch.float8_e4m3fn [M, C]) of src at its tensorwise scale, and 1 / scale (fp32 [1])."""
        M, C = src.shape
        dst = torch.empty((M, C), dtype=torch.float8_e4m3fn, device=src.device)
        inv = torch.empty((1,), dtype=torch.float32, device=src.device)
        scratch = torch.empty((lib().nc_op_fp8_scratch_bytes() // 4,), dtype=torch.float32, device=src.device)
        check(lib().nc_op_fp8_quantize(src.data_ptr(), int(src.dtype == torch.float32), M, C, _ptr(ssp), eps,
                                       dst.data_ptr(), inv.data_ptr(), scratch.data_ptr(), _stream_handle(None)),
              "nc_op_fp8_quantize")
        return dst, inv

    @staticmethod
    def gemm_fp8(A8, B8, inv_sa, inv_sb, epi="f32", cap=15.0, status=None):
        """epi((A8 . B8^T) * inv_sa * inv_sb) of e4m3 operands A8 [M, K], B8 [N, K]."""
        M, K = A8.shape
        N = B8.shape[0]
        dt = torch.bfloat16 if epi in ("bf16", "relu2_bf16", "softcap_bf16") else torch.float32
        out = torch.empty((M, N), dtype=dt, device=A8.device)
        check(lib().nc_op_gemm_fp8(A8.data_ptr(), B8.data_ptr(), M, N, K, EPI[epi], out.data_ptr(), N,
                                   inv_sa.data_ptr(), inv_sb.data_ptr(), cap, _ptr(status), _stream_handle(None)),
              "nc_op_gemm_fp8")
        return out

    @staticmethod
    def lmhead_ce_grad(xf, wlm, targets, lse, inv_count, ssp=None, C=0, eps=1e-6, cap=15.0, status=None):
        """bf16 [M, V]: rs * inv_count * (softmax(z) - onehot(target)) * (1 - (z/cap)^2)."""
        M, K = xf.shape
        V = wlm.shape[0]
        out = torch.empty((M, V), dtype=torch.bfloat16, device=xf.device)
        check(lib().nc_op_lmhead_ce_grad(xf.data_ptr(), wlm.data_ptr(), M, V, K, _ptr(ssp), eps, cap,
                                         targets.data_ptr(), lse.data_ptr(), inv_count.data_ptr(), out.data_ptr(), V,
                                         _ptr(status), _stream_handle(None)), "nc_op_lmhead_ce_grad")
        return out

    @staticmethod
    def mlp_hidden_grad(dy, w, h, ssp=None, eps=1e-6, status=None):
        """bf16 [M, F]: rs * (dy . w) * 2 sqrt(h), w the down projection's weight [C, F]."""
        M, C = dy.shape
        F = w.shape[1]
        out = torch.empty((M, F), dtype=torch.bfloat16, device=dy.device)
        check(lib().nc_op_mlp_hidden_grad(dy.data_ptr(), w.data_ptr(), M, F, C, _ptr(ssp), eps, h.data_ptr(),
                                          out.data_ptr(), _ptr(status), _stream_handle(None)), "nc_op_mlp_hidden_grad")
        return out

    @staticmethod
    def rms_backward(G, x, ssp, eps=1e-6, add=None):
        """Returns (dx fp32, dx bf16) = G - rs^2 x mean(G x) (+ add)."""
        M, C = G.shape
        dxf = torch.empty((M, C), dtype=torch.float32, device=G.device)
        dxb = torch.empty((M, C), dtype=torch.bfloat16, device=G.device)
        check(lib().nc_op_rms_backward(G.data_ptr(), x.data_ptr(), ssp.data_ptr(), _ptr(add), M, C, eps,
                                       dxf.data_ptr(), dxb.data_ptr(), _stream_handle(None)), "nc_op_rms_backward")
        return dxf, dxb

    @staticmethod
    def test_wait_timeout(A, B, out, limit_ns, skip_tile, status):
        """nc_op_test_wait_timeout: the bf16 GEMM with a short wait limit and one tile's accumulator
        signal withheld; returns the launch status code (the device status lands in `status`)."""
        M, K = A.shape
        N = B.shape[0]
        return lib().nc_op_test_wait_timeout(A.data_ptr(), B.data_ptr(), M, N, K, out.data_ptr(), out.shape[1],
                                             int(limit_ns), int(skip_tile), status.data_ptr(), _stream_handle(None))

    @staticmethod
    def gemm_residual(A, B, resid, a=1.0, b=0.0, Y=None, x_out=None, xm_out=None, status=None):
        """Returns (xb, ssp); x_out / xm_out are written in place when given."""
        M, K = A.shape
        N = B.shape[0]
        dev = A.device
        xb = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ssp = torch.empty((M, N // SS_GROUP), dtype=torch.float32, device=dev)
        check(lib().nc_op_gemm_residual(A.data_ptr(), B.data_ptr(), M, N, K, resid.data_ptr(), a, b, _ptr(Y),
                                        _ptr(x_out), _ptr(xm_out), xb.data_ptr(), ssp.data_ptr(), _ptr(status),
                                        _stream_handle(None)), "nc_op_gemm_residual")
        return xb, ssp

    @staticmethod
    def rope_table(T, D, base, device):
        """[D/2, T, 2] fp32 (cos, sin), position fastest."""
        t = torch.empty((D // 2, T, 2), dtype=torch.float32, device=device)
        check(lib().nc_op_rope_table(t.data_ptr(), T, D, base, _stream_handle(None)), "nc_op_rope_table")
        return t

    @staticmethod
    def qkv(xb, wqkv, T, H, Hkv, D, rope, eps, ssp, vgate=False, gate_scale=1.0, ve=None, tokens=None, V=0,
            status=None):
        """wqkv: the packed weight (see pack_qkv); vgate: it holds each kv head's gate rows."""
        M, C = xb.shape
        dev = xb.device
        q = torch.empty((M, H * D), dtype=torch.bfloat16, device=dev)
        k = torch.empty((M, Hkv * D), dtype=torch.bfloat16, device=dev)
        v = torch.empty((M, Hkv * D), dtype=torch.bfloat16, device=dev)
        check(lib().nc_op_qkv(xb.data_ptr(), wqkv.data_ptr(), M, T, C, H, Hkv, D, rope.data_ptr(), rope.shape[1],
                              eps, ssp.data_ptr(), int(bool(vgate)), gate_scale, _ptr(ve), _ptr(tokens), V,
                              q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(status), _stream_handle(None)),
              "nc_op_qkv")
        return q, k, v

    @staticmethod
    def pack_qkv(wq, wk, wv, wg=None, D=128):
        """The packed q|k|v weight nc_op_qkv takes: W_q, W_k, then W_v, or (wg [Hkv, c_g] given) for
        each kv head its D rows of W_v, its gate row (zero beyond c_g) and NC_QKV_GATE_ROWS - 1 zero rows."""
        if wg is None:
            return torch.cat([wq, wk, wv]).contiguous()
        Hkv, c_g = wg.shape
        C = wq.shape[1]
        parts = [wq, wk]
        for g in range(Hkv):
            gate = torch.zeros((QKV_GATE_ROWS, C), dtype=wq.dtype, device=wq.device)
            gate[0, :c_g] = wg[g]
            parts += [wv[g * D:(g + 1) * D], gate]
        return torch.cat(parts).contiguous()

    @staticmethod
    def attention(q, k, v, B, T, H, Hkv, D, window, status=None):
        y = torch.empty_like(q)
        check(lib().nc_op_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, T, H, Hkv, D, window, y.data_ptr(),
                                    _ptr(status), _stream_handle(None)), "nc_op_attention")
        return y

    @staticmethod
    def embed_smear(tokens, wte, smear_gate=None, c_s=0, embed_norm=False, eps=1e-6, a=1.0, status=None):
        """Returns (x0, x, xb, ssp)."""
        B, T = tokens.shape
        V, C = wte.shape
        dev = wte.device
        M = B * T
        x0 = torch.empty((M, C), dtype=torch.float32, device=dev)
        x = torch.empty((M, C), dtype=torch.float32, device=dev)
        xb = torch.empty((M, C), dtype=torch.bfloat16, device=dev)
        ssp = torch.empty((M, C // SS_GROUP), dtype=torch.float32, device=dev)
        check(lib().nc_op_embed_smear(tokens.data_ptr(), B, T, wte.data_ptr(), V, C, _ptr(smear_gate), c_s or C,
                                      int(embed_norm), eps, a, x0.data_ptr(), x.data_ptr(), xb.data_ptr(),
                                      ssp.data_ptr(), _ptr(status), _stream_handle(None)), "nc_op_embed_smear")
        return x0, x, xb, ssp

    @staticmethod
    def lmhead_ce(xf, wlm, targets, ssp=None, C=0, eps=1e-6, cap=15.0, status=None):
        """Cross-entropy partials of the soft-capped lm_head: returns (part [ceil(V/128), M], zt [M])."""
        M, K = xf.shape
        V = wlm.shape[0]
        part = torch.empty(((V + 127) // 128, M), dtype=torch.float32, device=xf.device)
        zt = torch.zeros((M,), dtype=torch.float32, device=xf.device)
        check(lib().nc_op_lmhead_ce(xf.data_ptr(), wlm.data_ptr(), M, V, K, _ptr(ssp), eps, cap, targets.data_ptr(),
                                    part.data_ptr(), zt.data_ptr(), _ptr(status), _stream_handle(None)),
              "nc_op_lmhead_ce")
        return part, zt

    @staticmethod
    def ce_finalize(part, zt, targets, V, token_bytes=None, status=None, with_lse=False):
        """Returns (loss [M], stats [2] = mean loss, bits per byte), and with with_lse also
        (lse [M], inv_count [1])."""
        M = zt.shape[0]
        dev = zt.device
        loss = torch.empty((M,), dtype=torch.float32, device=dev)
        stats = torch.empty((2,), dtype=torch.float32, device=dev)
        lse = torch.empty((M,), dtype=torch.float32, device=dev) if with_lse else None
        invc = torch.empty((1,), dtype=torch.float32, device=dev) if with_lse else None
        nbytes = lib().nc_op_ce_scratch_bytes(M)
        scratch = torch.empty((max(nbytes, 8) // 8,), dtype=torch.float64, device=dev)
        check(lib().nc_op_ce_finalize(part.data_ptr(), zt.data_ptr(), targets.data_ptr(), M, V, _ptr(token_bytes),
                                      loss.data_ptr(), stats.data_ptr(), scratch.data_ptr(), nbytes, _ptr(lse),
                                      _ptr(invc), _ptr(status), _stream_handle(None)), "nc_op_ce_finalize")
        return (loss, stats, lse, invc) if with_lse else (loss, stats)


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load ``libnc.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with decoder_only_forward_02_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class NcError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = f"{what}: {STATUS_NAMES.get(code, code)} ({lib().nc_status_string(code).decode()})"
        if code == 4:
            msg += f" [{lib().nc_last_cuda_error().decode()}]"
        super().__init__(msg)


def check(code: int, what: str) -> None:
    if code != NC_OK:
        raise NcError(code, what)


def _check_out(t: torch.Tensor, shape: tuple, dtype: torch.dtype, device, name: str) -> None:
    """A caller-provided output buffer must match exactly what the kernels write into it."""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous() or t.device != device:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_config(cfg, logits_bf16: bool = False, fp8: bool = False) -> tuple:
    """Build an NcConfig from any object with the model's attribute names (logits_bf16: the
    forward writes bf16 logits instead of fp32; fp8: the linear layers run on e4m3 copies).

    Returns (struct, keepalive) - the per-layer arrays must stay alive while the struct is used.
    """
    L = cfg.n_layer
    win = (ctypes.c_int * L)(*cfg.window_left)
    ve = (ctypes.c_ubyte * L)(*[1 if v else 0 for v in cfg.has_ve])
    c = NcConfig(
        n_layer=L, n_embd=cfg.n_embd, n_head=cfg.n_head, n_kv_head=cfg.n_kv_head, head_dim=cfg.head_dim,
        mlp_hidden=cfg.mlp_hidden, vocab_size=cfg.vocab_size, seq_len_ctx=cfg.seq_len_ctx,
        window_left=ctypes.cast(win, c_int_p), has_ve=ctypes.cast(ve, ctypes.POINTER(ctypes.c_ubyte)),
        use_smear=int(bool(cfg.use_smear)), use_backout=int(bool(cfg.use_backout)),
        embed_norm=int(bool(getattr(cfg, "embed_norm", False))),
        smear_gate_channels=int(getattr(cfg, "smear_gate_channels", 0)),
        ve_gate_channels=int(getattr(cfg, "ve_gate_channels", 0)),
        ve_gate_scale=float(getattr(cfg, "ve_gate_scale", 1.0)), rms_eps=float(getattr(cfg, "rms_eps", 1e-6)),
        rope_base=float(getattr(cfg, "rope_base", 10000.0)), softcap=float(getattr(cfg, "softcap", 15.0)),
        logits_bf16=int(bool(logits_bf16)), fp8=int(bool(fp8)))
    return c, (win, ve)


def packed_bytes(cfg) -> int:
    c, keep = make_config(cfg)
    n = ctypes.c_size_t()
    check(lib().nc_model_packed_bytes(ctypes.byref(c), ctypes.byref(n)), "nc_model_packed_bytes")
    return n.value


class Model:
    """A created nc_model.  ``weights``: dict of device bf16 tensors (names as in the weights
    layout: wte, wq.i, wk.i, wv.i, wo.i, wfc.i, wproj.i, ve.i, veg.i, smear, lm_head) plus the
    float lists resid_lambdas, x0_lambdas and the float backout_lambda."""

    def __init__(self, cfg, weights: Dict[str, object], device: Optional[torch.device] = None,
                 stream: Optional[torch.cuda.Stream] = None, logits_bf16: bool = False, fp8: bool = False):
        self.cfg = cfg
        self.device = torch.device(device) if device is not None else weights["wte"].device
        self.logits_dtype = torch.bfloat16 if logits_bf16 else torch.float32
        self._cstruct, self._keep = make_config(cfg, logits_bf16, fp8)
        L = cfg.n_layer

        def arr(name, optional=False):
            vals = []
            for i in range(L):
                t = weights.get(f"{name}.{i}")
                if t is None and not optional:
                    raise KeyError(f"{name}.{i}")
                vals.append(_ptr(t))
            return (ctypes.c_void_p * L)(*vals)

        self._arrays = {n: arr(n, optional=n in ("ve", "veg")) for n in
                        ("wq", "wk", "wv", "wo", "wfc", "wproj", "ve", "veg")}
        lr = (ctypes.c_float * L)(*weights["resid_lambdas"])
        l0 = (ctypes.c_float * L)(*weights["x0_lambdas"])
        self._lams = (lr, l0)
        self._weights = weights  # keep the device tensors alive
        w = NcWeights(
            wte=_ptr(weights["wte"]), lm_head=_ptr(weights["lm_head"]),
            smear_gate=_ptr(weights.get("smear")) if cfg.use_smear else None,
            resid_lambdas=ctypes.cast(lr, ctypes.POINTER(ctypes.c_float)),
            x0_lambdas=ctypes.cast(l0, ctypes.POINTER(ctypes.c_float)),
            backout_lambda=float(weights["backout_lambda"]),
            **{("ve_table" if k == "ve" else "ve_gate" if k == "veg" else k): ctypes.cast(v, c_void_pp)
               for k, v in self._arrays.items()})
        self._wstruct = w
        n = ctypes.c_size_t()
        check(lib().nc_model_packed_bytes(ctypes.byref(self._cstruct), ctypes.byref(n)), "nc_model_packed_bytes")
        self.packed = torch.empty(n.value, dtype=torch.uint8, device=self.device)
        h = ctypes.c_void_p()
        check(lib().nc_model_create(ctypes.byref(self._cstruct), ctypes.byref(w), self.packed.data_ptr(), n.value,
                                    _stream_handle(stream), ctypes.byref(h)), "nc_model_create")
        self.handle = h
        self._ws: Dict[tuple, torch.Tensor] = {}

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            try:
                lib().nc_model_destroy(h)
            except Exception:
                pass
            self.handle = None

    def workspace_bytes(self, B: int, T: int, host: bool = False, loss: bool = False) -> int:
        n = ctypes.c_size_t()
        fn = lib().nc_workspace_bytes_host if host else (lib().nc_workspace_bytes_loss if loss
                                                         else lib().nc_workspace_bytes)
        check(fn(self.handle, B, T, ctypes.byref(n)), "nc_workspace_bytes")
        return n.value

    def workspace(self, B: int, T: int, host: bool = False, loss: bool = False) -> torch.Tensor:
        key = (B, T, host, loss)
        if key not in self._ws:
            self._ws[key] = torch.empty(self.workspace_bytes(B, T, host, loss), dtype=torch.uint8,
                                        device=self.device)
        return self._ws[key]

    def forward(self, tokens: torch.Tensor, out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """tokens: device int32 [B, T] -> logits [B, T, V], fp32 or bf16 (logits_dtype; asynchronous)."""
        if tokens.dtype != torch.int32 or not tokens.is_cuda or not tokens.is_contiguous():
            raise ValueError("tokens must be a contiguous int32 CUDA tensor")
        B, T = tokens.shape
        V = self.cfg.vocab_size
        if out is None:
            out = torch.empty((B, T, V), dtype=self.logits_dtype, device=self.device)
        _check_out(out, (B, T, V), self.logits_dtype, tokens.device, "out")
        ws = self.workspace(B, T)
        check(lib().nc_forward(self.handle, tokens.data_ptr(), B, T, out.data_ptr(), ws.data_ptr(), ws.numel(),
                               _stream_handle(stream)), "nc_forward")
        return out

    def forward_loss(self, tokens: torch.Tensor, targets: torch.Tensor,
                     token_bytes: Optional[torch.Tensor] = None, loss: Optional[torch.Tensor] = None,
                     stats: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
        """tokens, targets: device int32 [B, T] (target < 0: ignored) -> (loss fp32 [B, T] in nats,
        stats fp32 [2] = mean loss, bits per byte); token_bytes: device int32 [V] or None.
        The lm_head is fused with the soft-cap and the cross-entropy: no logits are written."""
        for name, t in (("tokens", tokens), ("targets", targets)):
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
        if targets.shape != tokens.shape:
            raise ValueError("targets must have the shape of tokens")
        B, T = tokens.shape
        if loss is None:
            loss = torch.empty((B, T), dtype=torch.float32, device=self.device)
        if stats is None:
            stats = torch.empty((2,), dtype=torch.float32, device=self.device)
        _check_out(loss, (B, T), torch.float32, tokens.device, "loss")
        _check_out(stats, (2,), torch.float32, tokens.device, "stats")
        if token_bytes is not None:
            _check_out(token_bytes, (self.cfg.vocab_size,), torch.int32, tokens.device, "token_bytes")
        ws = self.workspace(B, T, loss=True)
        check(lib().nc_forward_loss(self.handle, tokens.data_ptr(), targets.data_ptr(), B, T, _ptr(token_bytes),
                                    loss.data_ptr(), stats.data_ptr(), ws.data_ptr(), ws.numel(),
                                    _stream_handle(stream)), "nc_forward_loss")
        return loss, stats

    def loss_grad_tail(self, tokens: torch.Tensor, targets: torch.Tensor,
                       token_bytes: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
        """nc_forward_loss_grad_tail: the loss path, then the gradient of the mean loss with respect to
        the lm_head and the last block's MLP down/up projections and attention output projection.
        Returns (stats fp32 [2], {"lm_head", "wproj", "wfc", "wo"}: fp32 gradients shaped like the
        weights)."""
        for name, t in (("tokens", tokens), ("targets", targets)):
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
        if targets.shape != tokens.shape:
            raise ValueError("targets must have the shape of tokens")
        B, T = tokens.shape
        c = self.cfg
        C, F, V, HD = c.n_embd, c.mlp_hidden, c.vocab_size, c.n_head * c.head_dim
        dev = self.device
        stats = torch.empty((2,), dtype=torch.float32, device=dev)
        g = {"lm_head": torch.empty((V, C), dtype=torch.float32, device=dev),
             "wproj": torch.empty((C, F), dtype=torch.float32, device=dev),
             "wfc": torch.empty((F, C), dtype=torch.float32, device=dev),
             "wo": torch.empty((C, HD), dtype=torch.float32, device=dev)}
        if token_bytes is not None:
            _check_out(token_bytes, (V,), torch.int32, tokens.device, "token_bytes")
        key = (B, T, "grad_tail")
        if key not in self._ws:
            n = ctypes.c_size_t()
            check(lib().nc_workspace_bytes_grad_tail(self.handle, B, T, ctypes.byref(n)), "nc_workspace_bytes_grad_tail")
            self._ws[key] = torch.empty(n.value, dtype=torch.uint8, device=dev)
        ws = self._ws[key]
        check(lib().nc_forward_loss_grad_tail(self.handle, tokens.data_ptr(), targets.data_ptr(), B, T,
                                              _ptr(token_bytes), stats.data_ptr(), g["lm_head"].data_ptr(),
                                              g["wproj"].data_ptr(), g["wfc"].data_ptr(), g["wo"].data_ptr(),
                                              ws.data_ptr(), ws.numel(), _stream_handle(stream)),
              "nc_forward_loss_grad_tail")
        return stats, g

    def kv_cache(self, B: int, T_max: int) -> torch.Tensor:
        """A device buffer for the KV cache of B rows and up to T_max positions."""
        n = ctypes.c_size_t()
        check(lib().nc_kv_cache_bytes(self.handle, B, T_max, ctypes.byref(n)), "nc_kv_cache_bytes")
        return torch.empty(n.value, dtype=torch.uint8, device=self.device)

    def prefill(self, tokens: torch.Tensor, cache: torch.Tensor, T_max: int, out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """tokens: device int32 [B, T] -> logits [B, T, V] (logits_dtype); fills the cache with positions 0..T-1."""
        if tokens.dtype != torch.int32 or not tokens.is_cuda or not tokens.is_contiguous():
            raise ValueError("tokens must be a contiguous int32 CUDA tensor")
        B, T = tokens.shape
        if out is None:
            out = torch.empty((B, T, self.cfg.vocab_size), dtype=self.logits_dtype, device=self.device)
        _check_out(out, (B, T, self.cfg.vocab_size), self.logits_dtype, tokens.device, "out")
        ws = self.workspace(B, T)
        check(lib().nc_prefill(self.handle, tokens.data_ptr(), B, T, cache.data_ptr(), cache.numel(), T_max,
                               out.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(stream)), "nc_prefill")
        return out

    def decode_step(self, prev_tokens: torch.Tensor, tokens: torch.Tensor, pos: int, cache: torch.Tensor,
                    T_max: int, out: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """tokens / prev_tokens: device int32 [B] (positions pos and pos - 1) -> logits [B, V] (logits_dtype) of
        position pos; appends the new keys and values to the cache."""
        for name, t in (("tokens", tokens), ("prev_tokens", prev_tokens)):
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
        B = tokens.shape[0]
        if prev_tokens.shape != tokens.shape or tokens.dim() != 1:
            raise ValueError("tokens and prev_tokens must both have shape [B]")
        if out is None:
            out = torch.empty((B, self.cfg.vocab_size), dtype=self.logits_dtype, device=self.device)
        _check_out(out, (B, self.cfg.vocab_size), self.logits_dtype, tokens.device, "out")
        key = ("decode", B)
        if key not in self._ws:
            n = ctypes.c_size_t()
            check(lib().nc_workspace_bytes_decode(self.handle, B, ctypes.byref(n)), "nc_workspace_bytes_decode")
            self._ws[key] = torch.empty(n.value, dtype=torch.uint8, device=self.device)
        ws = self._ws[key]
        check(lib().nc_decode_step(self.handle, prev_tokens.data_ptr(), tokens.data_ptr(), B, pos, cache.data_ptr(),
                                   cache.numel(), T_max, out.data_ptr(), ws.data_ptr(), ws.numel(),
                                   _stream_handle(stream)), "nc_decode_step")
        return out

    def forward_host(self, tokens: torch.Tensor, out: torch.Tensor,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """tokens: host int32 [B, T] (pinned for full speed) -> out: host [B, T, V] (logits_dtype);
        synchronous."""
        B, T = tokens.shape
        _check_out(out, (B, T, self.cfg.vocab_size), self.logits_dtype, torch.device("cpu"), "out")
        ws = self.workspace(B, T, host=True)
        check(lib().nc_forward_host(self.handle, tokens.data_ptr(), B, T, out.data_ptr(), ws.data_ptr(),
                                    ws.numel(), _stream_handle(stream)), "nc_forward_host")
        return out

    def status(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        """Synchronise and return (and clear) the device status code."""
        return lib().nc_get_status(self.handle, _stream_handle(stream))

    def timing(self, enable: bool) -> None:
        check(lib().nc_timing_enable(self.handle, int(enable)), "nc_timing_enable")

    def timing_read(self) -> Dict[str, tuple]:
        out = {}
        for k, name in enumerate(KERNEL_CLASSES):
            ms = ctypes.c_double()
            n = ctypes.c_int()
            check(lib().nc_timing_read(self.handle, k, ctypes.byref(ms), ctypes.byref(n)), "nc_timing_read")
            out[name] = (ms.value, n.value)
        return out

    def grad_tail_launch_count(self) -> int:
        return lib().nc_grad_tail_launch_count(self.handle)

    def launch_count(self, loss: bool = False, kv: bool = False) -> int:
        fn = lib().nc_forward_loss_launch_count if loss else (lib().nc_kv_launch_count if kv
                                                              else lib().nc_forward_launch_count)
        return fn(self.handle)
