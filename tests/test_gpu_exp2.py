"""The softmax warps' FMA-pipe exp2 (range reduction + fitted degree-3 polynomial)
against CUDA's exp2, within the fit's relative-error bound (GPU)."""
import pytest
import torch

import transformer_self_attention_gb300 as tsa

pytestmark = pytest.mark.gpu


def _poly(x):
    y = torch.empty_like(x)
    st = tsa.attn_selftest_exp2(x.data_ptr(), y.data_ptr(), x.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == tsa.ATTN_OK
    torch.cuda.synchronize()
    return y


def test_exp2_poly_relative_error_on_the_softmax_range():
    g = torch.Generator(device="cpu").manual_seed(5)
    x = torch.cat([torch.linspace(-125.0, 9.0, 1 << 20), torch.rand(1 << 18, generator=g) * 134 - 125,
                   torch.tensor([0.0, -0.5, 0.5, -1.0, 1.0, 8.0, -124.5, -125.0])]).float().cuda()
    y = _poly(x)
    ref = torch.exp2(x.double())              # CUDA's exp2, in double
    rel = ((y.double() - ref) / ref).abs().max().item()
    assert rel <= 1e-4, rel                   # the fit's float32 bound is 7.5e-5


def test_exp2_poly_clamps_below_minus_125():
    x = torch.tensor([-126.0, -200.0, -1e30], device="cuda")
    y = _poly(x)
    assert bool((y > 0).all()) and bool((y <= 2.0 ** -124).all())


def test_exp2_poly_odd_length():
    x = torch.linspace(-3, 3, 7, device="cuda")
    assert torch.allclose(_poly(x).double(), torch.exp2(x.double()), rtol=1e-4, atol=0)
