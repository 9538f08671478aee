"""GPU parity of the KV-cache quantization against the oracle: after every
append, the quantized store (codes, binary32 scale bits, zero points) and the
cache as read back must equal the oracle's bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from activation_quantization_quantize_b300 import inputs, qlin

pytestmark = pytest.mark.gpu


def kv_inputs(T, C, seed):
    k = inputs.normal((T, C), 1.0, seed)
    inputs.outlier_channels(k, max(1, C // 64), 10.0, 30.0, seed + 1)   # K's outliers sit in channels
    v = inputs.normal((T, C), 1.0, seed + 2)
    return torch.from_numpy(k).to(torch.bfloat16), torch.from_numpy(v).to(torch.bfloat16)


def unpack(codes, n, bits):
    a = codes.cpu().numpy()
    if bits == 4:
        return oracle.unpack_nibbles(a, n, False)
    return a.astype(np.int32)


def check(cache, k, v, G, R, D, bits):
    T = cache.c.length
    kh, vh = k[:T].float().numpy(), v[:T].float().numpy()
    ref = oracle.kv_cache_reference(kh, vh, G, R, D, bits)
    assert cache.c.quantized == ref["tq"]
    kr, vr = cache.read()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(kr.float().cpu().numpy(), oracle.round_bf16(ref["k_hat"]))
    np.testing.assert_array_equal(vr.float().cpu().numpy(), oracle.round_bf16(ref["v_hat"]))
    tq, C = ref["tq"], kh.shape[1]
    if tq:
        kc, ks, kz, vc, vs, vz = cache.state()
        np.testing.assert_array_equal(unpack(kc, tq * C, bits).reshape(tq, C), ref["k_codes"])
        np.testing.assert_array_equal(ks.cpu().numpy().view(np.uint32).reshape(-1, C),
                                      ref["k_scale"].view(np.uint32))
        np.testing.assert_array_equal(kz.cpu().numpy().reshape(-1, C), ref["k_zero"])
        np.testing.assert_array_equal(unpack(vc, tq * C, bits).reshape(tq, C), ref["v_codes"])
        np.testing.assert_array_equal(vs.cpu().numpy().view(np.uint32).reshape(tq, -1),
                                      ref["v_scale"].view(np.uint32))
        np.testing.assert_array_equal(vz.cpu().numpy().reshape(tq, -1), ref["v_zero"])


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("G,R", [(32, 48), (128, 128), (16, 0)])
def test_kv_cache_appends_match_the_oracle(bits, G, R):
    """A prefill, then decode appends of 1, 5, G + 3 and G tokens; the state
    and the read-back cache are checked after every append."""
    C, D = 512, 128
    T_total = 700
    k, v = kv_inputs(T_total, C, seed=bits + G + R)
    cache = qlin.KVCache(capacity=((T_total + G - 1) // G) * G, channels=C, head_dim=D, group=G, residual=R,
                         bits=bits)
    kd, vd = k.cuda(), v.cuda()
    sizes = [300, 1, 1, 5, G + 3, G, 1, 1, 17, 100, 1]
    t = 0
    for n in sizes:
        cache.append(kd[t:t + n], vd[t:t + n])
        t += n
        check(cache, k, v, G, R, D, bits)
    while t < T_total:                                   # the rest one token at a time, checked every 37
        cache.append(kd[t:t + 1], vd[t:t + 1])
        t += 1
        if t % 37 == 0 or t == T_total:
            check(cache, k, v, G, R, D, bits)
    assert qlin.qlin_device_error() == 0


def test_kv_cache_window_and_capacity():
    C, D, G, R = 256, 64, 32, 64
    k, v = kv_inputs(200, C, seed=5)
    cache = qlin.KVCache(capacity=192, channels=C, head_dim=D, group=G, residual=R, bits=4)
    kd, vd = k.cuda(), v.cuda()
    cache.append(kd[:R + G - 1], vd[:R + G - 1])           # still inside the window
    assert cache.c.quantized == 0
    check(cache, k, v, G, R, D, 4)
    cache.append(kd[R + G - 1:R + G], vd[R + G - 1:R + G])  # the first group leaves it
    assert cache.c.quantized == G
    check(cache, k, v, G, R, D, 4)
    with pytest.raises(qlin.QlinError):
        cache.append(kd[:200 - (R + G) + 1], vd[:200 - (R + G) + 1])   # would pass the capacity of 192
    assert cache.c.length == R + G                         # a refused call changes nothing
