"""C-ABI checks that need no GPU: the library loads, exports every declared symbol, and the
host-side validation returns the documented status codes before touching the device."""
import ctypes
import os
import re
from dataclasses import replace

import pytest

from decoder_only_forward_02_b300 import binding as B
from synth import get_workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in ("nc.h", "nc_ops.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        names += re.findall(r"^NC_API\s+[\w\s\*]+?\b(nc_\w+)\s*\(", src, flags=re.M)
    return names


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    names = _declared()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B._SIGS)   # and the binding gives every entry point its signature


def test_status_strings():
    lib = B.lib()
    for code in range(7):
        assert lib.nc_status_string(code)
    assert lib.nc_status_string(99) == b"unknown status"


def _packed(cfg):
    c, keep = B.make_config(cfg)
    n = ctypes.c_size_t()
    return B.lib().nc_model_packed_bytes(ctypes.byref(c), ctypes.byref(n)), n.value


def test_packed_bytes_formula():
    cfg = get_workload("d12").model
    code, n = _packed(cfg)
    assert code == 0
    # q|k|v rows per layer, plus, on the 6 value-embedding layers, 16 rows per kv head (its gate row
    # and 15 zero rows)
    qkv = (12 * (6 + 12) * 128 + 6 * 6 * 16) * 768 * 2
    rope = 2048 * 64 * 8
    assert n == 256 + rope + qkv


@pytest.mark.parametrize("change,code", [
    (dict(n_embd=640), 1),           # C != H*D
    (dict(n_kv_head=4), 1),          # H % Hkv != 0
    (dict(head_dim=96, n_embd=576), 2),
    (dict(mlp_hidden=3000), 2),
    (dict(vocab_size=32769), 2),
    (dict(smear_gate_channels=6), 2),
    (dict(ve_gate_channels=1000), 1),
    (dict(ve_gate_channels=12), 2),  # c_g must be a multiple of 8 (nc.h)
    (dict(n_layer=0, window_left=(), has_ve=()), 1),
])
def test_config_validation(change, code):
    cfg = replace(get_workload("d12").model, **change)
    assert _packed(cfg)[0] == code


def test_null_arguments_rejected_without_device_work():
    lib = B.lib()
    c, keep = B.make_config(get_workload("tiny").model)
    n = ctypes.c_size_t()
    assert lib.nc_model_packed_bytes(None, ctypes.byref(n)) == 1
    assert lib.nc_model_packed_bytes(ctypes.byref(c), None) == 1
    h = ctypes.c_void_p(1)
    assert lib.nc_model_create(ctypes.byref(c), None, None, 0, None, ctypes.byref(h)) == 1
    assert h.value is None
    assert lib.nc_forward(None, None, 1, 1, None, None, 0, None) == 1
    assert lib.nc_forward_host(None, None, 1, 1, None, None, 0, None) == 1
    assert lib.nc_workspace_bytes(None, 1, 1, ctypes.byref(n)) == 1
    assert lib.nc_get_status(None, None) == 1
    assert lib.nc_timing_enable(None, 1) == 1
    assert lib.nc_forward_launch_count(None) == 0
    lib.nc_model_destroy(None)
    # per-kernel entry points validate before launching
    assert lib.nc_op_gemm(None, None, 1, 32, 64, 0, None, 32, None, 0, 1e-6, 15.0, None, None) == 1
    assert lib.nc_op_gemm_residual(None, None, 1, 128, 64, None, 1.0, 0.0, None, None, None, None, None, None,
                                   None) == 1
    assert lib.nc_op_attention(None, None, None, 1, 1, 1, 1, 128, -1, None, None, None) == 1
    assert lib.nc_op_rope_table(None, 4, 8, 1e4, None) == 1
    assert lib.nc_op_embed_smear(None, 1, 1, None, 1, 128, None, 0, 0, 1e-6, 1.0, None, None, None, None, None,
                                 None) == 1
    assert lib.nc_op_lmhead_ce(None, None, 1, 32, 64, None, 1e-6, 15.0, None, None, None, None, None) == 1
    assert lib.nc_op_ce_finalize(None, None, None, 1, 32, None, None, None, None, 0, None, None, None, None) == 1
    assert lib.nc_op_ce_scratch_bytes(0) == 0 and lib.nc_op_ce_scratch_bytes(300) >= 16
    assert lib.nc_forward_loss(None, None, None, 1, 1, None, None, None, None, 0, None) == 1
    assert lib.nc_forward_loss_launch_count(None) == 0
    assert lib.nc_kv_launch_count(None) == 0
    assert lib.nc_kv_cache_bytes(None, 1, 1, None) == 1
    assert lib.nc_prefill(None, None, 1, 1, None, 0, 1, None, None, 0, None) == 1
    assert lib.nc_decode_step(None, None, None, 1, 1, None, 0, 2, None, None, 0, None) == 1
    assert lib.nc_workspace_bytes_grad_tail(None, 1, 1, ctypes.byref(n)) == 1
    assert lib.nc_forward_loss_grad_tail(None, None, None, 1, 1, None, None, None, None, None, None, None, 0,
                                         None) == 1
    assert lib.nc_grad_tail_launch_count(None) == 0


def test_kernel_class_names():
    lib = B.lib()
    assert [lib.nc_kernel_class_name(i).decode() for i in range(13)] == B.KERNEL_CLASSES
    assert lib.nc_kernel_class_name(13) == b"unknown"


def test_headers_are_plain_c_and_link(tmp_path):
    """The boundary is a C ABI: both headers compile as pedantic C99 and as C++, and a C program
    links against the library and calls its host-only entry points."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_nc.c"
    src.write_text(
        '#include "nc.h"\n#include "nc_ops.h"\n#include <string.h>\n'
        "int main(void) {\n"
        '  if (strcmp(nc_status_string(NC_ERR_WORKSPACE), "buffer smaller than required") != 0) return 1;\n'
        "  if (nc_forward_launch_count(0) != 0 || nc_op_ce_scratch_bytes(0) != 0) return 2;\n"
        "  size_t n = 0;\n"
        "  if (nc_model_packed_bytes(0, &n) != NC_ERR_INVALID_ARG) return 3;\n"
        "  return 0;\n}\n")
    inc = os.path.join(ROOT, "include")
    lib = os.path.dirname(B.LIB_PATH)
    exe = tmp_path / "use_nc"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, str(src), "-o", str(exe),
                    "-L", lib, "-lnc", f"-Wl,-rpath,{lib}"], check=True, capture_output=True)
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", "-I", inc, "-x", "c++", "-fsyntax-only", str(src)],
                   check=True, capture_output=True)
    assert subprocess.run([str(exe)]).returncode == 0


def test_output_buffer_checks():
    import torch
    dev = torch.device("cpu")
    ok = torch.empty((2, 3), dtype=torch.float32)
    B._check_out(ok, (2, 3), torch.float32, dev, "out")
    for bad in (torch.empty((3, 2), dtype=torch.float32), torch.empty((2, 3), dtype=torch.float64),
                torch.empty((3, 2), dtype=torch.float32).t()):
        with pytest.raises(ValueError):
            B._check_out(bad, (2, 3), torch.float32, dev, "out")


def test_loss_ops_validate_before_launch():
    """Every case here fails validation, so nothing is launched (fake pointers are never used)."""
    lib = B.lib()
    a = 4096   # an aligned address that is never dereferenced
    # nc_op_lmhead_ce(xf, wlm, M, V, C, ssp, eps, cap, targets, part, zt, status, stream)
    assert lib.nc_op_lmhead_ce(a + 8, a, 4, 64, 64, None, 1e-6, 15.0, a, a, a, None, None) == 1    # misaligned xf
    assert lib.nc_op_lmhead_ce(a, a, 4, 64, 64, None, 1e-6, 0.0, a, a, a, None, None) == 1        # cap <= 0
    assert lib.nc_op_lmhead_ce(a, a, 4, 48, 64, None, 1e-6, 15.0, a, a, a, None, None) == 2       # V % 32
    assert lib.nc_op_lmhead_ce(a, a, 4, 64, 96, None, 1e-6, 15.0, a, a, a, None, None) == 2       # C % 64
    assert lib.nc_op_lmhead_ce(a, a, 4, 64, 64, a, 1e-6, 15.0, a, a, a, None, None) == 1          # ssp, C % 128
    # nc_op_ce_finalize(part, zt, targets, M, V, token_bytes, loss, stats, scratch, bytes, lse, inv_count,
    #                   status, stream)
    need = lib.nc_op_ce_scratch_bytes(300)
    assert lib.nc_op_ce_finalize(a, a, a, 300, 64, None, None, a, a, need - 8, None, None, None, None) == 3
    assert lib.nc_op_ce_finalize(a, a, a, 300, 64, None, None, a, a + 4, need, None, None, None, None) == 1
    assert lib.nc_op_ce_finalize(a, a, a, 0, 64, None, None, a, a, need, None, None, None, None) == 1     # M < 1
    assert lib.nc_op_ce_finalize(a, a, a, 300, 64, None, None, a, a, need, a + 2, None, None, None) == 1  # lse


def test_backward_ops_validate_before_launch():
    """Every case here fails validation, so nothing is launched (fake pointers are never used)."""
    lib = B.lib()
    a = 4096
    # nc_op_gemm_t(A, B, M, N, K, a_mn, b_mn, epi, out, ldo, ssp, C, eps, cap, split_ws, bytes, status, stream)
    assert lib.nc_op_gemm_t(a, a, 64, 64, 64, 2, 0, 7, a, 64, None, 0, 1e-6, 15.0, None, 0, None, None) == 1   # a_mn not 0/1
    assert lib.nc_op_gemm_t(a, a, 64, 64, 60, 0, 1, 7, a, 64, None, 0, 1e-6, 15.0, None, 0, None, None) == 2   # K % 8, K-major A
    assert lib.nc_op_gemm_t(a, a, 60, 64, 64, 1, 1, 7, a, 64, None, 0, 1e-6, 15.0, None, 0, None, None) == 2   # M % 8, MN-major A
    assert lib.nc_op_gemm_t(a, a, 64, 48, 64, 1, 1, 7, a, 64, None, 0, 1e-6, 15.0, None, 0, None, None) == 2   # N % 32
    assert lib.nc_op_gemm_t(a, a, 64, 64, 64, 1, 1, 7, a, 32, None, 0, 1e-6, 15.0, None, 0, None, None) == 1   # ldo < N
    assert lib.nc_op_gemm_t(a, a, 64, 64, 64, 1, 1, 5, a, 64, None, 0, 1e-6, 15.0, None, 0, None, None) == 1   # epilogue kind
    assert lib.nc_op_gemm_t(a + 8, a, 64, 64, 64, 1, 1, 7, a, 64, None, 0, 1e-6, 15.0, None, 0, None, None) == 1
    assert lib.nc_op_gemm_t(a, a, 64, 64, 64, 1, 1, 0, a, 64, None, 0, 1e-6, 15.0, a, 1 << 20, None, None) == 1  # split, bf16
    assert lib.nc_op_gemm_t(a, a, 64, 64, 64, 1, 1, 7, a, 64, None, 0, 1e-6, 15.0, a + 4, 1 << 20, None, None) == 1
    assert lib.nc_op_gemm_split_ws_bytes(0, 64, 64, 64) == 0
    # nc_op_lmhead_ce_grad(xf, wlm, M, V, C, ssp, eps, cap, targets, lse, inv_count, out, ldo, status, stream)
    assert lib.nc_op_lmhead_ce_grad(a, a, 4, 64, 64, None, 1e-6, 15.0, a, a, None, a, 64, None, None) == 1  # inv_count
    assert lib.nc_op_lmhead_ce_grad(a, a, 4, 64, 64, None, 1e-6, 0.0, a, a, a, a, 64, None, None) == 1      # cap
    assert lib.nc_op_lmhead_ce_grad(a, a, 4, 64, 64, None, 1e-6, 15.0, a, a, a, a, 60, None, None) == 1     # ldo
    assert lib.nc_op_lmhead_ce_grad(a, a, 4, 48, 64, None, 1e-6, 15.0, a, a, a, a, 48, None, None) == 2     # V % 32
    # nc_op_mlp_hidden_grad(dy, w, M, F, C, ssp, eps, h, out, status, stream)
    assert lib.nc_op_mlp_hidden_grad(a, a, 4, 64, 128, None, 1e-6, None, a, None, None) == 1   # h missing
    assert lib.nc_op_mlp_hidden_grad(a, a, 4, 48, 128, None, 1e-6, a, a, None, None) == 2      # F % 32
    assert lib.nc_op_mlp_hidden_grad(a, a, 4, 64, 100, None, 1e-6, a, a, None, None) == 2      # C % 8
    # nc_op_rms_backward(G, x, ssp, add, M, C, eps, dx_f32, dx_b16, stream)
    assert lib.nc_op_rms_backward(a, a, a, None, 4, 128, 1e-6, None, None, None) == 1          # no output
    assert lib.nc_op_rms_backward(a, a, a, None, 4, 192, 1e-6, a, None, None) == 2             # C % 128
    assert lib.nc_op_rms_backward(a, a, a, None, 4, 4096, 1e-6, a, None, None) == 2            # C > 2048
    assert lib.nc_op_rms_backward(a + 4, a, a, None, 4, 128, 1e-6, a, None, None) == 1         # misaligned G
