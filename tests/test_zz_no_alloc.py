"""qlin_quantize_noalloc: the quantizer for callers that cannot allocate
device memory (e.g. a plug-in whose host framework owns all device memory,
or code that runs under an allocator's lock).  It uses the library's fixed
scratch array instead of a caller workspace; its results must equal
qlin_quantize's, call after call, through the C ABI.

This file is collected last so that a failure here leaves every other test
already run."""
import ctypes as C

import numpy as np
import pytest
import torch

from activation_quantization_quantize_b300 import inputs, qlin

pytestmark = pytest.mark.gpu


def _outputs(p, rows, cols, dev):
    code4 = p.code in (qlin.QLIN_S4, qlin.QLIN_U4)
    q = torch.full((rows, cols // 2 if code4 else cols), 0x5A, dtype=torch.uint8, device=dev)
    ns = qlin.num_scopes(p, rows, cols)
    s = torch.full((ns,), 7.0, dtype=torch.float16 if p.scale_dtype == qlin.QLIN_F16 else torch.float32,
                   device=dev)
    z = torch.full((ns,), 99, dtype=torch.int32, device=dev)
    return q, s, z


CASES = [("s8", "tensor", 0, 0.0), ("u8", "col", 0, 0.0), ("s8", "tensor", 0, 99.9),
         ("u4", "group", 64, 0.0), ("s8", "row", 0, 0.0)]


@pytest.mark.parametrize("code,gran,group,pct", CASES)
def test_noalloc_matches_workspace_entry_point(code, gran, group, pct):
    dev = torch.device("cuda", 0)
    rows, cols = 257, 1024
    lib = qlin.load()
    for call in range(2):   # two calls in a row: the shared scratch must not leak state
        x = torch.from_numpy(inputs.normal((rows, cols), 1.0 + call, 300 + call)).to(torch.bfloat16).to(dev)
        p = qlin.make_params(code, gran, group=group, percentile=pct)
        q1, s1, z1 = _outputs(p, rows, cols, dev)
        q2, s2, z2 = _outputs(p, rows, cols, dev)
        zp1 = None if p.symmetric else z1
        zp2 = None if p.symmetric else z2
        nbytes = qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, rows, cols, 0, p)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.qlin_quantize(x.data_ptr(), qlin.QLIN_BF16, rows, cols, cols, None, C.byref(p), q1.data_ptr(),
                               s1.data_ptr(), None if zp1 is None else zp1.data_ptr(),
                               ws.data_ptr() if nbytes else None, nbytes, stream)
        assert rc == qlin.QLIN_OK
        rc = lib.qlin_quantize_noalloc(x.data_ptr(), qlin.QLIN_BF16, rows, cols, cols, None, C.byref(p),
                                       q2.data_ptr(), s2.data_ptr(), None if zp2 is None else zp2.data_ptr(),
                                       stream)
        assert rc == qlin.QLIN_OK
        torch.cuda.synchronize()
        assert torch.equal(q1, q2)
        assert torch.equal(s1, s2)
        if not p.symmetric:
            assert torch.equal(z1, z2)
    assert qlin.qlin_device_error() == 0


@pytest.mark.parametrize("code,asym", [("s4", False), ("u4", True)])
def test_noalloc_many_groups_needs_no_scratch(code, asym):
    """A 4096 x 4096 weight in groups of 128 (131,072 groups, the W4A16 decode
    weight): row-local scopes keep their statistics on chip, so the call needs
    none of the scratch, succeeds and matches qlin_quantize, twice in a row."""
    dev = torch.device("cuda", 0)
    rows, cols = 4096, 4096
    lib = qlin.load()
    p = qlin.make_params(code, "group", group=128, scale_f16=True)
    assert qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, rows, cols, 0, p) == 0
    for call in range(2):
        w = torch.from_numpy(inputs.normal((rows, cols), 0.02 * (1 + call), 310 + call)).to(torch.bfloat16).to(dev)
        q1, s1, z1 = qlin.quantize(w, p)
        q2, s2, z2 = _outputs(p, rows, cols, dev)
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.qlin_quantize_noalloc(w.data_ptr(), qlin.QLIN_BF16, rows, cols, cols, None, C.byref(p),
                                       q2.data_ptr(), s2.data_ptr(), z2.data_ptr() if asym else None, stream)
        assert rc == qlin.QLIN_OK
        torch.cuda.synchronize()
        assert torch.equal(q1.view(torch.uint8), q2)
        assert torch.equal(s1, s2)
        if asym:
            assert torch.equal(z1, z2)
    assert qlin.qlin_device_error() == 0


def test_noalloc_rejects_oversized_scratch():
    lib = qlin.load()
    p = qlin.make_params("s8", "col")
    cols = 65536 + 8          # per-column statistics need 8 bytes per column
    assert qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, 4, cols, 0, p) > 512 * 1024
    fake = C.c_void_p(0x10000)  # validation fails before any pointer is used
    rc = lib.qlin_quantize_noalloc(fake, qlin.QLIN_BF16, 4, cols, cols, None, C.byref(p), fake, fake, None, None)
    assert rc == qlin.QLIN_ERR_WORKSPACE
