"""The fixed-order sum kernel of the data-parallel gradient exchange
(ll_sum_ordered): bitwise the ascending-order FP32 additions, for FP32 and
16-bit tables (FP32 accumulation, one rounding), aligned and unaligned
rows."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ascending(parts):
    acc = parts[0].float().clone()
    for k in range(1, parts.shape[0]):
        acc += parts[k].float()
    return acc.to(parts.dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("k,n,pad", [(1, 5, 0), (2, 1000003, 0), (5, 4099, 3), (8, 1 << 20, 0)])
def test_sum_ordered_is_the_ascending_sum(lib, dtype, k, n, pad):
    g = torch.Generator(device="cuda")
    g.manual_seed(k * 7 + n)
    buf = torch.randn(k, n + pad, generator=g, device="cuda").to(dtype)
    parts = buf[:, :n]
    out = lib.sum_ordered(parts)
    torch.cuda.synchronize()
    assert lib.check_status() == 0
    want = _ascending(parts)
    bits = torch.int32 if dtype == torch.float32 else torch.int16
    assert torch.equal(out.view(bits), want.view(bits))


def test_sum_ordered_rejects_overlap_and_bad_shapes(lib):
    L = lib.load()
    buf = torch.zeros(3, 64, device="cuda")
    # out inside the parts
    assert L.ll_sum_ordered(lib._ptr(buf), 3, 64, 64, lib.LL_F32, lib._ptr(buf[1]),
                            lib._stream()) == 1
    # ld < n
    out = torch.empty(64, device="cuda")
    assert L.ll_sum_ordered(lib._ptr(buf), 3, 64, 32, lib.LL_F32, lib._ptr(out),
                            lib._stream()) == 3
    # n == 0: nothing to do
    assert L.ll_sum_ordered(None, 0, 0, 0, lib.LL_F32, None, lib._stream()) == 0
