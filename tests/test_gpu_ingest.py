"""moe_mx_blocks_unpack: 17-byte MXFP4 checkpoint blocks -> canonical codes and scales, bit for bit
against the oracle's definition, for both nibble orders."""
import numpy as np
import pytest
import torch

import oracle

from gpu_support import device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__ as g
    g.build_cuda()
    import block_scaled_fp4_sqrt_gb300 as m
    return m


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("n", [1, 33, 10007])
def test_unpack_matches_oracle(moe, split, n):
    rng = np.random.default_rng(n + split)
    blocks = rng.integers(0, 256, size=(n, 17), dtype=np.uint8)
    codes, scales = moe.moe_mx_blocks_unpack(torch.from_numpy(blocks).to(device()),
                                             moe.MOE_MX_NIBBLES_SPLIT if split else moe.MOE_MX_NIBBLES_PAIRED)
    torch.cuda.synchronize()
    want_c, want_s = oracle.mx_blocks_unpack(blocks, split)
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(scales.cpu().numpy(), want_s)


def test_unpack_to_unaligned_output(moe):
    rng = np.random.default_rng(5)
    n = 100
    blocks = torch.from_numpy(rng.integers(0, 256, size=(n, 17), dtype=np.uint8)).to(device())
    out = torch.zeros(16 * n + 1, dtype=torch.uint8, device=device())
    sc = torch.zeros(n, dtype=torch.uint8, device=device())
    L = moe.lib()
    import ctypes
    st = L.moe_mx_blocks_unpack(ctypes.c_void_p(blocks.data_ptr()), n, moe.MOE_MX_NIBBLES_SPLIT,
                                ctypes.c_void_p(out.data_ptr() + 1), ctypes.c_void_p(sc.data_ptr()), None)
    torch.cuda.synchronize()
    assert st == 0
    want_c, want_s = oracle.mx_blocks_unpack(blocks.cpu().numpy(), True)
    assert np.array_equal(out[1:].cpu().numpy().reshape(n, 16), want_c)
    assert out[0].item() == 0


def test_unpack_rejects_bad_arguments(moe):
    with pytest.raises(moe.MoEError):
        moe.moe_mx_blocks_unpack(torch.zeros(17, dtype=torch.uint8, device=device()), 7)
