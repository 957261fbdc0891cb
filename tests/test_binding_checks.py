"""The Python binding checks dtypes, shapes and devices before a pointer reaches the library
(the kernels trust the sizes passed beside the pointers).  CPU tensors suffice: each call
below fails in the check, before any launch."""
import pytest
import torch

from mixture_experts_layer_scores_b300 import moe

bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32


def z(*shape, dt=bf):
    return torch.zeros(*shape, dtype=dt)


@pytest.mark.parametrize("call, err, what", [
    (lambda: moe.moe_permute(z(4, 64), z(4, 2, dt=torch.int64), 8), TypeError, "topk_idx"),
    (lambda: moe.moe_permute(z(3, 64), z(4, 2, dt=i32), 8), ValueError, "xn"),
    (lambda: moe.moe_permute(z(4, 64), z(4, 2, dt=i32), 8, counts=z(9, dt=i32)), ValueError, "counts"),
    (lambda: moe.moe_permute(z(4, 64), z(4, 2, dt=i32), 8, x_perm=z(8, 64, dt=f32)), TypeError, "x_perm"),
    (lambda: moe.moe_unpermute_combine(z(8, 64), z(4, 2, dt=i32), z(4, 2, dt=torch.float64)), TypeError,
     "topk_gate"),
    (lambda: moe.moe_unpermute_combine(z(8, 64), z(4, 2, dt=i32), z(4, 2, dt=f32), residual=z(4, 32)),
     ValueError, "residual"),
    (lambda: moe.moe_grouped_swiglu(z(16, 64), z(3, dt=i32), z(2, 128, 64), z(2, 128, 64), z(2, 128, 64)),
     ValueError, "w_down"),
    (lambda: moe.moe_grouped_swiglu(z(16, 64), z(2, dt=i32), z(2, 128, 64), z(2, 128, 64), z(2, 64, 128)),
     ValueError, "offsets"),
    (lambda: moe.moe_grouped_swiglu_gather(z(4, 64), z(8, dt=torch.int64), z(3, dt=i32), z(2, 128, 64),
                                           z(2, 128, 64), z(2, 64, 128)), TypeError, "perm_token"),
    (lambda: moe.moe_router_topk_split(z(4, 64, dt=f32), z(3, 8, 64), z(8, dt=f32), 2), TypeError, "xn"),
    (lambda: moe.moe_router_topk(z(4, 64), z(8, 64, dt=bf), z(8, dt=f32), 2), TypeError, "w_router"),
    (lambda: moe.moe_bias_update(z(8, dt=torch.int64), z(8, dt=f32), 16, 1e-3), TypeError, "counts"),
    (lambda: moe.moe_bias_update(z(8, dt=i32), z(7, dt=f32), 16, 1e-3), ValueError, "bias"),
])
def test_bad_argument_rejected_before_launch(call, err, what):
    with pytest.raises(err, match=what):
        call()
