"""GPU checks of the host-buffer runtime (fa_host_plan_create / fa_host_step /
fa_host_wait): several steps with different host inputs in flight at once
give, bit for bit, what fa_forward + fa_backward give on device copies of the
same inputs; the plan owns its device memory and leaves the caller's device
and streams alone."""
import pytest
import torch

from fa_inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 300, 64, True), (2, 3, 1000, 128, False),
                                            (1, 4, 2048, 128, True)])
def test_host_steps_equal_device_calls(fa, B, H, N, d, causal):
    steps = 5
    ins = [make_inputs(B, H, N, d, seed=100 + i) for i in range(steps)]
    pinned_in = [[t.pin_memory() for t in step] for step in ins]
    outs = [[torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory() for _ in range(4)]
            + [torch.empty((B, H, N), dtype=torch.float32).pin_memory()] for _ in range(steps)]
    plan = fa.HostPlan(B, H, N, d, causal=causal)
    for (q, k, v, dO), (o, dq, dk, dv, lse) in zip(pinned_in, outs):
        plan.step(q, k, v, dO, o, lse, dq, dk, dv)
    plan.wait()
    plan.close()
    dev = torch.device("cuda")
    for (q, k, v, dO), (o, dq, dk, dv, lse) in zip(ins, outs):
        qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
        o_r, lse_r = fa.fa_forward(qd, kd, vd, causal=causal)
        dq_r, dk_r, dv_r = fa.fa_backward(qd, kd, vd, o_r, dOd, lse_r, causal=causal)
        torch.cuda.synchronize()
        for got, ref in ((o, o_r), (lse, lse_r), (dq, dq_r), (dk, dk_r), (dv, dv_r)):
            assert torch.equal(got, ref.cpu())


def test_host_plan_frees_its_memory(fa):
    torch.cuda.synchronize()
    before = torch.cuda.mem_get_info()[0]
    plan = fa.HostPlan(2, 8, 4096, 128, causal=True)
    during = torch.cuda.mem_get_info()[0]
    plan.close()
    after = torch.cuda.mem_get_info()[0]
    per_slot = 8 * 2 * 8 * 4096 * 128 * 2
    assert before - during >= 2 * per_slot  # two slots of eight tensors at least
    assert abs(after - before) < 64 << 20
