"""kv_quant_pack on the GPU against the oracle quantiser: bit-exact codes, scales, zeros."""
import numpy as np
import pytest
import torch

from bit_mixed_precision_gb300 import inputs, kvq
from oracle import quant as OQ
from tests.helpers import u16, u32

pytestmark = pytest.mark.gpu

AX = {kvq.AXIS_CHANNEL: "channel", kvq.AXIS_TOKEN: "token"}


def _x(B, H, T, D, dtype, seed, scale=10.0):
    x = inputs.make_qkv(B, H, H, T, D, dtype=dtype, seed=seed,
                        outliers=inputs.outlier_channels(H, D, 3, seed), outlier_scale=scale)
    return x.k


def _compare(got, ref):
    codes, s, z = got
    oc, os_, oz = ref
    assert np.array_equal(u32(codes), oc.view(np.uint32)), "codes"
    assert np.array_equal(u16(s), os_.view(np.uint16)), "scales"
    assert np.array_equal(u16(z), oz.view(np.uint16)), "zeros"


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("axis", [kvq.AXIS_CHANNEL, kvq.AXIS_TOKEN])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_bit_exact(bits, axis, dtype):
    x = _x(2, 3, 96, 128, dtype, seed=bits + 10 * axis)
    got = kvq.kv_quant_pack(x.cuda(), bits, 32, axis)
    ref = OQ.kv_quant_pack(x.float().numpy(), bits, 32, AX[axis])
    _compare(got, ref)


@pytest.mark.parametrize("group", [16, 32, 64])
def test_pack_group_sizes(group):
    x = _x(1, 2, 128, 64, torch.float16, seed=group)
    for axis in (kvq.AXIS_CHANNEL, kvq.AXIS_TOKEN):
        _compare(kvq.kv_quant_pack(x.cuda(), 2, group, axis),
                 OQ.kv_quant_pack(x.float().numpy(), 2, group, AX[axis]))


def test_pack_gather():
    """Selected (ascending, gappy) positions are packed in list order."""
    B, H, T, D, n = 2, 2, 300, 128, 64
    x = _x(B, H, T, D, torch.float16, seed=3)
    r = np.random.default_rng(0)
    idx = np.stack([np.stack([np.sort(r.choice(T, n, replace=False)) for _ in range(H)])
                    for _ in range(B)]).astype(np.int32)
    gi = torch.from_numpy(idx).cuda()
    for axis in (kvq.AXIS_CHANNEL, kvq.AXIS_TOKEN):
        _compare(kvq.kv_quant_pack(x.cuda(), 2, 32, axis, gather_idx=gi),
                 OQ.kv_quant_pack(x.float().numpy(), 2, 32, AX[axis], gather_idx=idx))
    assert kvq.device_status() == 0


def test_pack_edge_values():
    """Constant groups, exact zeros and signed zeros, tiny values."""
    B, H, T, D = 1, 1, 64, 128
    x = torch.zeros((B, H, T, D), dtype=torch.float16)
    x[0, 0, :, 1] = 0.5                         # constant channel
    x[0, 0, 5, 2] = -0.0
    x[0, 0, :, 3] = torch.linspace(-1e-6, 1e-6, T).to(torch.float16)   # subnormal range
    x[0, 0, 7, :] = 1.0                         # constant token row
    x[0, 0, 9, 64:] = -65504.0 / 4
    for axis in (kvq.AXIS_CHANNEL, kvq.AXIS_TOKEN):
        for bits in (2, 4, 8):
            _compare(kvq.kv_quant_pack(x.cuda(), bits, 32, axis),
                     OQ.kv_quant_pack(x.float().numpy(), bits, 32, AX[axis]))


def test_pack_empty():
    x = _x(1, 1, 32, 128, torch.float16, seed=1).cuda()
    codes, s, z = kvq.kv_quant_pack(x, 2, 32, kvq.AXIS_TOKEN, n=0)
    assert codes.numel() == 0
    torch.cuda.synchronize()


def test_pack_bad_gather_index_is_reported():
    """An out-of-range position is skipped on the device and reported, not a fault."""
    x = _x(1, 1, 64, 128, torch.float16, seed=2).cuda()
    gi = torch.arange(32, dtype=torch.int32, device="cuda").reshape(1, 1, 32).clone()
    gi[0, 0, 5] = 64
    kvq.kv_quant_pack(x, 2, 32, kvq.AXIS_TOKEN, gather_idx=gi)
    assert kvq.device_status() == kvq.KVQ_EDEVICE
    assert kvq.device_status() == 0             # reading clears it
