"""Failure detection on the GPU without a fault: the pipelined kernels'
bounded waits.

qlin_debug_stall_producers(1, limit) makes the copy-issuing roles of the
tensor-core GEMMs and of the streamed per-token quantizer issue nothing (a
flag that nothing ever sets, from the waiters' point of view) and lowers the
wait limit.  Each kernel must then give up on its own, report
QLIN_ERR_TIMEOUT through qlin_device_error, free its TMEM and leave the
context usable: the next normal call on the same device must be bit-exact
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from activation_quantization_quantize_b300 import inputs, qlin
from helpers import GEMM_REL_TOL, codes_to_int, host_f32, oracle_quantize, rel_err_out, scales_f32

pytestmark = pytest.mark.gpu

LIMIT = 200_000   # SM cycles (~0.1 ms) before a wait gives up


class stalled:
    def __enter__(self):
        assert qlin.qlin_device_error() == qlin.QLIN_OK
        qlin.qlin_debug_stall_producers(True, LIMIT)

    def __exit__(self, *exc):
        qlin.qlin_debug_stall_producers(False)
        return False


def _w8a8_inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    qx = torch.from_numpy(rng.integers(-127, 128, (M, K)).astype(np.int8)).cuda()
    qw = torch.from_numpy(rng.integers(-127, 128, (N, K)).astype(np.int8)).cuda()
    sx = torch.from_numpy(rng.uniform(0.001, 0.1, M).astype(np.float32)).cuda()
    sw = torch.from_numpy(rng.uniform(0.001, 0.1, N).astype(np.float32)).cuda()
    return qx, sx, qw, sw


@pytest.mark.parametrize("kernel", ["pair", "tc1"])
def test_w8a8_wait_times_out_then_recovers(kernel, monkeypatch):
    """Both tensor-core kernels: the CTA pair (converters stall, the drain
    monitor's wait runs out) and the single CTA (the TMA warp stalls)."""
    monkeypatch.setenv("QLIN_W8A8_KERNEL", kernel)
    M, N, K = 256, 512, 2048
    qx, sx, qw, sw = _w8a8_inputs(M, N, K, 1)
    with stalled():
        qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.float32)
        assert qlin.qlin_device_error() == qlin.QLIN_ERR_TIMEOUT
    assert qlin.qlin_device_error() == qlin.QLIN_OK          # the word was read and cleared
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = qlin.gemm_w8a8(qx, sx, qw, sw, out_dtype=torch.bfloat16, acc_out=acc)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == qlin.QLIN_OK
    acco = oracle.w8a8_acc(qx.cpu().numpy(), qw.cpu().numpy())
    np.testing.assert_array_equal(acc.cpu().numpy(), acco)
    yo = oracle.w8a8_out(acco, sx.cpu().numpy(), sw.cpu().numpy())
    assert rel_err_out(host_f32(y), yo) < GEMM_REL_TOL


@pytest.mark.parametrize("M", [64, 256])
def test_w4a16_wait_times_out_then_recovers(M):
    """M = 64: the TMEM-operand kernel; M = 256: the shared-memory-operand one."""
    N, K = 512, 2048
    w = torch.from_numpy(inputs.normal((N, K), 0.02, 3)).to(torch.bfloat16).cuda()
    x = torch.from_numpy(inputs.normal((M, K), 1.0, 4)).to(torch.bfloat16).cuda()
    p = qlin.make_params("u4", "group", group=128, scale_f16=True)
    q, s, z = qlin.quantize(w, p)
    packed, hdr = qlin.pack_w4(q, s, z, N, K, 128)
    with stalled():
        qlin.gemm_w4a16(x, packed, hdr)
        assert qlin.qlin_device_error() == qlin.QLIN_ERR_TIMEOUT
    y = qlin.gemm_w4a16(x, packed, hdr)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == qlin.QLIN_OK
    what = oracle.w4_dequant(codes_to_int(q, p, N, K), scales_f32(s), z.cpu().numpy(), 128)
    yo = oracle.matmul_f64(host_f32(x), what)
    assert rel_err_out(host_f32(y), yo) < GEMM_REL_TOL


@pytest.mark.parametrize("kernel", ["reg", "smem"])
@pytest.mark.parametrize("gran,cols", [("row", 28672), ("row", 4096), ("group", 4096)])
def test_streamed_quantize_wait_times_out_then_recovers(kernel, gran, cols, monkeypatch):
    """Per-token rows of 28672 and 4096 and per-group-128 rows of 4096 bf16
    values stream through shared memory by bulk copies (the chunks held in
    registers, or read from the row buffer; 512, 64 and 128 threads); with
    the copies held back every CTA's wait runs out."""
    if kernel == "smem":
        monkeypatch.setenv("QLIN_QROW", "smem")
    if cols == 28672:
        rows = 300
        x = inputs.downproj_activation(rows, outliers=True).cuda()
    else:
        rows = 600
        x = torch.from_numpy(inputs.normal((rows, cols), 1.0, 5)).to(torch.bfloat16).cuda()
    p = qlin.make_params("s8", gran, group=128 if gran == "group" else 0)
    with stalled():
        qlin.quantize(x, p)
        assert qlin.qlin_device_error() == qlin.QLIN_ERR_TIMEOUT
    q, s, _ = qlin.quantize(x, p)
    torch.cuda.synchronize()
    assert qlin.qlin_device_error() == qlin.QLIN_OK
    qo, so, _ = oracle_quantize(host_f32(x), p)
    np.testing.assert_array_equal(codes_to_int(q, p, rows, cols), qo)
    np.testing.assert_array_equal(scales_f32(s).view(np.uint32), so.view(np.uint32))


def test_stall_hook_rejects_a_non_positive_limit():
    with pytest.raises(qlin.QlinError):
        qlin.qlin_debug_stall_producers(True, 0)
