"""Plans (one captured graph) over INT4 and FP8 projections, fused and alone,
mixed with BF16 ones, and the full decode step with quantised weights, against
the CPU oracles, every element."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs, workloads
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"
W4, F8, BF = binding.GEMV_WEIGHT_INT4, binding.GEMV_WEIGHT_FP8, binding.GEMV_WEIGHT_BF16


def ref_quant(kind, Wq, S, x, K, rows=None):
    Wh, Sh = Wq.cpu().numpy(), S.cpu()
    if rows is not None:
        Wh = Wh[rows]
        Sh = Sh[rows]
    if kind == F8:
        return oracle.gemv_fp8(Wh, Sh.numpy(), inputs.bits(x), K, threads=oracle.default_threads())
    return oracle.gemv_w4(Wh, inputs.bits(Sh), inputs.bits(x), K, threads=oracle.default_threads())


def test_mixed_quant_plan():
    K, B = 4096, 1
    xh = inputs.activations(B, K, seed=1, device=DEV)
    xi = inputs.activations(B, 14336, seed=2, device=DEV)
    projs, checks = [], []

    def add(kind, N, Kp, x, group, seed, eps=None):
        y = torch.full((B, N), float("nan"), device=DEV)
        if kind == F8:
            W, S = inputs.fp8_weight(N, Kp, seed=seed, device=DEV)
            lds = 0
        elif kind == W4:
            W, S = inputs.w4_weight_device(N, Kp, seed=seed, device=DEV)
            lds = S.shape[1]
        else:
            W, S, lds = inputs.weight(N, Kp, seed=seed, device=DEV), None, 0
        projs.append((W, x, y, N, Kp, W.shape[1], B, group, eps, False, kind, S, lds))
        checks.append((kind, W, S, x, y, Kp, eps))

    for nm, n in (("q", 4096), ("k", 1024), ("v", 1024)):
        add(F8, n, K, xh, 1, 10 + n, eps=1e-5)          # fused FP8 QKV with the RMSNorm prologue
    add(F8, 4096, K, xh, 0, 20)                         # o_proj alone
    add(W4, 14336, K, xh, 2, 21)                        # fused INT4 gate/up
    add(W4, 14336, K, xh, 2, 22)
    add(BF, 4096, 14336, xi, 0, 23)                     # a BF16 down projection between them
    add(W4, 4096, 14336, xi, 0, 24)                     # and an INT4 one
    plan = binding.Plan(projs)
    assert plan.num_launches() == 5
    s = torch.cuda.Stream()
    plan.capture(s)
    for _ in range(2):
        for c in checks:
            c[4].fill_(float("nan"))
        torch.cuda.synchronize()
        plan.launch(s)
        s.synchronize()
        for kind, W, S, x, y, Kp, eps in checks:
            if kind == BF:
                y_ref, sc = gu.reference(W, x, Kp)
            else:
                y_ref, sc = ref_quant(kind, W, S, x, Kp)
            if eps is not None:
                xd = x.double().cpu().numpy()
                r = 1.0 / np.sqrt(np.mean(xd * xd, axis=1) + eps)
                y_ref, sc = y_ref * r[:, None], sc * r[:, None]
            gu.assert_parity(y.cpu().numpy(), y_ref, sc, f"kind={kind} N={W.shape[0]}")
    plan.destroy()


def test_quant_plan_rejects_bad_projections():
    K = 4096
    x = inputs.activations(1, K, seed=1, device=DEV)
    y = torch.empty((1, 64), device=DEV)
    W, S = inputs.fp8_weight(64, K, seed=1, device=DEV)
    for bad in [(W, x, y, 64, K, W.shape[1], 1, 0, None, True, F8, S, 0),      # stream-K on FP8
                (W, x, y, 64, 100, W.shape[1], 1, 0, None, False, F8, S, 0),   # K not a multiple of 64
                (W, x, y, 64, K, W.shape[1], 1, 0, None, False, 7, S, 0)]:     # unknown kind
        with pytest.raises(binding.GemvError):
            binding.Plan([bad])


@pytest.mark.parametrize("weights", ["fp8", "int4"])
def test_full_quant_decode_step_every_element(weights):
    """The full step with quantised weights in the benchmark's configuration:
    one graph of 129 launches, the RMSNorm prologue on QKV, gate/up and the LM
    head. Every output of every projection against the oracle."""
    free, _ = torch.cuda.mem_get_info()
    if free < 24 << 30:
        pytest.skip("needs 24 GB of free device memory")
    step = workloads.DecodeStep(workloads.decode_step_spec(), seed=0, device=DEV, weights=weights)
    plan = step.plan(rms_eps=1e-5)
    assert plan.num_launches() == 32 * 4 + 1
    s = torch.cuda.Stream()
    plan.capture(s)
    for y in step.outputs():
        y.fill_(float("nan"))
    torch.cuda.synchronize()
    plan.launch(s)
    s.synchronize()
    kind = F8 if weights == "fp8" else W4
    checked = 0
    for p in step.projs:
        yh = p.y.cpu().numpy()
        y_ref, sc = ref_quant(kind, p.W, p.S, p.x, p.K)
        normed = p.name.endswith(("q_proj", "k_proj", "v_proj", "gate_proj", "up_proj")) or p.name == "lm_head"
        if normed:
            xd = p.x.double().cpu().numpy()
            r = 1.0 / np.sqrt(np.mean(xd * xd, axis=1) + 1e-5)
            y_ref, sc = y_ref * r[:, None], sc * r[:, None]
        gu.assert_parity(yh, y_ref, sc, p.name)
        checked += p.N
    assert checked == 1_504_512
    plan.destroy()
    del step
    torch.cuda.empty_cache()
