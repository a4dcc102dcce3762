"""EmuLinear on the GPU: the nn.Linear drop-in of the blog post's TF32x3
section (trained weights, bias and shapes kept; FP32 in and out; the gradient
with respect to the layer input also through the emulated GEMM, because
forces are derivatives of the energy).  Each product is checked against the
oracle's FP64 GEMM with the element-wise bound; a small energy model is
checked end to end (energy and forces) against float64 PyTorch on the CPU."""
import numpy as np
import pytest

import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def emu():
    return emu_module()


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_forward_and_gradients_match_the_oracle(emu, mode):
    import torch
    from fp32_emulated_gemm_split_gb300.linear import EmuLinear
    torch.manual_seed(0)
    lin = EmuLinear(256, 192, device="cuda", mode=mode)
    r = W.rng(5)
    x_np = W.normal(r, (4, 300, 256))
    g_np = W.normal(r, (4, 300, 192))
    x = torch.from_numpy(x_np).cuda().requires_grad_(True)
    y = lin(x)
    y.backward(torch.from_numpy(g_np).cuda())
    torch.cuda.synchronize()
    Wt = lin.weight.detach().cpu().numpy()
    b = lin.bias.detach().cpu().numpy()
    X2, G2 = x_np.reshape(-1, 256), g_np.reshape(-1, 192)
    bmode = "tf32x3" if mode == "tf32x3" else "bf16x9"
    # forward: y = x W^T + b  (bias enters as beta * C with beta = 1)
    C0 = np.broadcast_to(b, (X2.shape[0], 192)).astype(np.float32).copy()
    Cref, Sabs = oracle.gemm_ref(X2, Wt, transB=True, beta=1.0, C0=C0)
    assert checks.error_ratio(y.detach().cpu().numpy().reshape(-1, 192), Cref, Sabs, 256, 1.0, 1.0,
                              C0, mode=bmode) <= 1.0
    # input gradient: dx = dy W
    Cref, Sabs = oracle.gemm_ref(G2, Wt)
    assert checks.error_ratio(x.grad.cpu().numpy().reshape(-1, 256), Cref, Sabs, 192, 1.0, 0.0,
                              mode=bmode) <= 1.0
    # weight gradient: dW = dy^T x
    Cref, Sabs = oracle.gemm_ref(G2, X2, transA=True)
    assert checks.error_ratio(lin.weight.grad.cpu().numpy(), Cref, Sabs, X2.shape[0], 1.0, 0.0,
                              mode=bmode) <= 1.0
    assert np.allclose(lin.bias.grad.cpu().numpy(), G2.astype(np.float64).sum(0), rtol=1e-5, atol=1e-4)


def test_swapped_energy_model_energy_and_forces(emu):
    """A small MLP energy model: E = sum(MLP(positions-derived features));
    forces = -dE/dx.  The emulated model must match float64 at least as well
    as the FP32 model run by PyTorch (cuBLAS FP32 without TF32)."""
    import torch
    from fp32_emulated_gemm_split_gb300.linear import swap_linear_layers
    torch.manual_seed(1)
    torch.backends.cuda.matmul.allow_tf32 = False

    def make():
        return torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.SiLU(),
                                   torch.nn.Linear(256, 256), torch.nn.SiLU(),
                                   torch.nn.Linear(256, 1))

    ref64 = make().double()
    fp32 = make().cuda()
    fp32.load_state_dict({k: v.float() for k, v in ref64.state_dict().items()})
    emu_model = make().cuda()
    emu_model.load_state_dict({k: v.float() for k, v in ref64.state_dict().items()})
    swap_linear_layers(emu_model, mode="bf16x9")
    assert sum(isinstance(m, torch.nn.Linear) for m in emu_model.modules()) == 0

    x64 = torch.from_numpy(W.normal(W.rng(9), (4096, 64)).astype(np.float64)).requires_grad_(True)
    e64 = ref64(x64).sum()
    (f64,) = torch.autograd.grad(-e64, x64)

    def energy_forces(model):
        x = x64.detach().float().cuda().requires_grad_(True)
        e = model(x).sum()
        (f,) = torch.autograd.grad(-e, x)
        return e.double().item(), f.double().cpu()

    e_emu, f_emu = energy_forces(emu_model)
    e_32, f_32 = energy_forces(fp32)
    err = lambda f: float(torch.linalg.norm(f - f64) / torch.linalg.norm(f64))  # noqa: E731
    assert abs(e_emu - e64.item()) <= 1e-5 * abs(e64.item()) + 1e-4
    assert err(f_emu) <= 2e-6
    # the emulated forces are not worse than FP32's by more than rounding noise
    assert err(f_emu) <= 2 * err(f_32) + 1e-7


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_weight_pieces_follow_the_weight(emu, mode):
    """The layer keeps its weight's split pieces between calls and remakes
    them after an in-place update (an optimiser step) or a new weight: the
    output always matches the current weight, bit for bit the same as
    emu_sgemm on it, and the forward product runs no split kernel once the
    pieces exist."""
    import torch
    from fp32_emulated_gemm_split_gb300.linear import EmuLinear
    torch.manual_seed(3)
    lin = EmuLinear(256, 256, bias=False, device="cuda", mode=mode)
    x = torch.randn(12288, 256, device="cuda")

    def direct():
        return emu.emu_sgemm(x, lin.weight.detach(), transB=True, mode=mode)

    with torch.no_grad():
        y0 = lin(x)
        assert torch.equal(y0, direct())
        emu.emu_profile_enable(True)
        y1 = lin(x)                                  # pieces reused
        torch.cuda.synchronize()
        n_split = emu.emu_profile_read("split")[0]
        emu.emu_profile_enable(False)
        assert torch.equal(y1, y0)
        if mode == "bf16x9":
            assert n_split == 0                      # one fused launch, A split on chip
        lin.weight.mul_(0.5)                         # in place: the version changes
        y2 = lin(x)
        assert torch.equal(y2, direct())
        assert not torch.equal(y2, y0)
        lin.weight = torch.nn.Parameter(torch.randn(256, 256, device="cuda"))
        y3 = lin(x)
        assert torch.equal(y3, direct())
