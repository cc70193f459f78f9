"""GPU parity of the INT8 checkpoint store/load (the infra page's section 6.6.2)
against the oracle: codes, scales and dequantised rows bit for bit (both sides
decide the codes with correctly rounded fp32 division and ties-to-even), pairs
with invalid indices skipped, every other byte untouched."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import kda_ckpt_load_int8, kda_ckpt_store_int8
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import bytes_of, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


def crafted_ties(D, dtype):
    """A [D][D] block whose columns have amax = 127 / 64 (scale 2^-6 exactly) and other
    entries at (n + 1/2) 2^-6: every code is a rounding tie (exact in fp32 and bf16)."""
    v = torch.arange(D, dtype=torch.float32).unsqueeze(1)
    k = torch.arange(D, dtype=torch.float32).unsqueeze(0)
    x = (((v * 7 + k * 3) % 201) - 100 + 0.5) * 2.0 ** -6
    x[0, :] = 127 * 2.0 ** -6
    x[1, ::2] = -127 * 2.0 ** -6
    return x.to(dtype)


@pytest.mark.parametrize("D,H", [(128, 3), (64, 2), (32, 4)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("itype", [torch.int32, torch.int64])
def test_int8_store_load_bit_exact(D, H, dtype, itype):
    N, slots = 8, 6
    P = H * D * D
    pc = wl.paged_cache(N, H, D, D, dtype, P + 64, seed=D + H, device=DEV)
    # varied column magnitudes, an all-zero column block, and a block of rounding ties
    mag = torch.exp(torch.randn(N, H, 1, D, generator=wl.generator(3, DEV), device=DEV) * 2).to(dtype)
    pc.view.mul_(mag)
    pc.view[2, 0, :, : D // 2] = 0
    pc.view[5, H - 1] = crafted_ties(D, dtype).to(DEV)
    src = torch.tensor([5, 2, -1, 7, 0, 3], dtype=itype)
    dst = torch.tensor([1, 4, 0, 9, 2, -2], dtype=itype)   # pairs 2 (src -1), 3 (slot 9), 5 (slot -2): skipped
    q = torch.full((slots, H, D, D), 55, dtype=torch.int8, device=DEV)
    sc = torch.full((slots, H, D), -1.0, dtype=torch.float32, device=DEV)
    kda_ckpt_store_int8(pc.view, src.to(DEV), dst.to(DEV), q, sc)
    torch.cuda.synchronize()
    host = raw(pc.backing)
    body = np.ascontiguousarray(host[pc.front:pc.front + N * pc.row_stride])
    q_ref = np.full((slots, H, D, D), 55, dtype=np.int8)
    sc_ref = np.full((slots, H, D), -1.0, dtype=np.float32)
    oracle.ckpt_store_int8(body, N, pc.row_stride, H, D, D, src.numpy(), dst.numpy(), q_ref, sc_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
    # load slots back into a second cache (sentinel-filled), rows 6, 1, 3; slot 7 and row -1 invalid
    pc2 = wl.paged_cache(N, H, D, D, dtype, P + 64, seed=0, device=DEV, fill=False)
    before2 = raw(pc2.backing)
    lsrc = torch.tensor([1, 4, 2, 7, 1], dtype=itype)
    ldst = torch.tensor([6, 1, 3, 0, -1], dtype=itype)
    kda_ckpt_load_int8(q, sc, lsrc.to(DEV), pc2.view, ldst.to(DEV))
    torch.cuda.synchronize()
    body2 = np.ascontiguousarray(before2[pc2.front:pc2.front + N * pc2.row_stride])
    oracle.ckpt_load_int8(q_ref, sc_ref, lsrc.numpy(), ldst.numpy(), body2, N, pc2.row_stride, H, D, D)
    want = before2.copy()
    want[pc2.front:pc2.front + N * pc2.row_stride] = body2
    np.testing.assert_array_equal(bytes_of(pc2.backing), want.view(np.uint8))


def test_int8_round_trip_error_is_half_a_step():
    """Store then load: |x' - x| <= scale / 2 per element (the quantisation bound)."""
    N, H, D = 4, 2, 128
    pc = wl.paged_cache(N, H, D, D, torch.float32, None, seed=11, device=DEV)
    idx = torch.arange(N, dtype=torch.int32, device=DEV)
    q = torch.empty(N, H, D, D, dtype=torch.int8, device=DEV)
    sc = torch.empty(N, H, D, dtype=torch.float32, device=DEV)
    kda_ckpt_store_int8(pc.view, idx, idx, q, sc)
    back = wl.paged_cache(N, H, D, D, torch.float32, None, seed=0, device=DEV, fill=False)
    kda_ckpt_load_int8(q, sc, idx, back.view, idx)
    torch.cuda.synchronize()
    err = (back.view - pc.view).abs()
    assert torch.all(err <= sc.unsqueeze(2) * (0.5 + 1e-5))
    amax = pc.view.abs().amax(dim=2)
    assert torch.allclose(sc, amax / 127, rtol=1e-6)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_int8_store_subnormal_scales(dtype):
    """Columns whose amax / 127 is 0 or subnormal get scale 0 and codes 0 on both sides;
    columns just above the smallest normal scale keep the ordinary rule; bit for bit."""
    H, D = 1, 32
    tiny = float(torch.finfo(torch.float32).tiny)  # 2^-126
    x = torch.randn(D, D, generator=wl.generator(5, "cpu"))
    x[:, 0] = x[:, 0].sign() * 1e-45                # subnormal values: amax / 127 -> 0
    x[:, 1] = x[:, 1] / x[:, 1].abs().max() * 100 * tiny  # amax = 100 * 2^-126: amax / 127 subnormal
    x[:, 2] = x[:, 2] * 1e-40
    x[:, 3] = torch.linspace(-1, 1, D) * 127 * tiny * 2  # amax / 127 = 2^-125, normal
    x[:, 4] = 0.0
    x = x.to(dtype).float()  # the values the cache holds
    pc = wl.paged_cache(2, H, D, D, dtype, None, seed=1, device=DEV)
    pc.view[1, 0] = x.to(dtype).to(DEV)
    idx = torch.tensor([1], dtype=torch.int32, device=DEV)
    q = torch.full((1, H, D, D), 55, dtype=torch.int8, device=DEV)
    sc = torch.full((1, H, D), -1.0, dtype=torch.float32, device=DEV)
    kda_ckpt_store_int8(pc.view, idx, torch.zeros_like(idx), q, sc)
    torch.cuda.synchronize()
    host = raw(pc.backing)
    body = np.ascontiguousarray(host[pc.front:pc.front + 2 * pc.row_stride])
    q_ref = np.full((1, H, D, D), 55, dtype=np.int8)
    sc_ref = np.full((1, H, D), -1.0, dtype=np.float32)
    oracle.ckpt_store_int8(body, 2, pc.row_stride, H, D, D, [1], [0], q_ref, sc_ref)
    assert np.all(sc_ref[0, 0, [0, 1, 2, 4]] == 0.0) and sc_ref[0, 0, 3] > 0.0
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
