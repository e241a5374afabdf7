"""Host logic of the fused backward pass (CPU, no GPU): every group steps exactly once per
backward, when its last gradient has been accumulated, with the gradients autograd produced,
and the gradients are released afterwards."""
import torch

from memory_lean_optimizer_gb300.hooks import FusedStepper, split_groups


class FakeGroup:
    def __init__(self, params, log):
        self.params = params
        self.log = log

    def step(self, grads, hp, stream):
        self.log.append(([p for p in self.params], [g.clone() for g in grads]))


def test_split_groups_balanced_and_ordered():
    params = [torch.empty(n) for n in (10, 10, 10, 10, 100, 5, 5)]
    idx = split_groups(params, 3)
    assert [i for g in idx for i in g] == list(range(len(params)))
    assert len(idx) == 3 and all(len(g) > 0 for g in idx)
    assert split_groups(params, 100) == [[i] for i in range(len(params))]
    assert split_groups(params, 1) == [list(range(len(params)))]


def test_each_group_steps_once_with_autograd_grads():
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(8, 16), torch.nn.ReLU(), torch.nn.Linear(16, 4))
    ref = torch.nn.Sequential(torch.nn.Linear(8, 16), torch.nn.ReLU(), torch.nn.Linear(16, 4))
    ref.load_state_dict(model.state_dict())
    log = []
    stepper = FusedStepper(list(model.parameters()), 2, {}, lambda ps: FakeGroup(ps, log))
    x = torch.randn(5, 8)
    for it in range(2):
        log.clear()
        model(x).pow(2).sum().backward()
        ref.zero_grad()
        ref(x).pow(2).sum().backward()
        assert len(log) == 2                                   # two groups, one step each
        stepped = [id(p) for ps, _ in log for p in ps]
        assert sorted(stepped) == sorted(id(p) for p in model.parameters())
        ref_grads = {name: p.grad for name, p in ref.named_parameters()}
        names = {id(p): n for n, p in model.named_parameters()}
        for ps, gs in log:
            for p, g in zip(ps, gs):
                assert torch.equal(g, ref_grads[names[id(p)]])
        assert all(p.grad is None for p in model.parameters())  # released after the step
    stepper.remove()
    model(x).sum().backward()
    assert all(p.grad is not None for p in model.parameters())
