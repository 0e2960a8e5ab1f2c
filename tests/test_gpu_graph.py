"""Decode steps captured in a CUDA graph: pop_decode_step and pop_moe_decode_step allocate nothing and
never synchronize, so a sequence of steps can be captured once and replayed. Replays must give the
same bits as the same steps run eagerly (the kernels reduce in a fixed order)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import online_structured_ffn_gb300 as pop
    torch.cuda.set_device(0)
    return pop, torch, torch.device("cuda", 0)


def up(env, a):
    _, torch, dev = env
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def _layer(env, D, N, B, period):
    pop = env[0]
    Wg, W1, W2 = synth.ffn_weights(0, D, N)
    return pop.PopFFN(up(env, Wg), up(env, W1), up(env, W2), r=0.3, gamma=0.1, period=period, max_batch=B)


@pytest.mark.parametrize("B,period", [(1, 1), (16, 1), (16, 4), (64, 2)])
def test_decode_steps_replay_from_a_graph(env, B, period):
    _, torch, dev = env
    D, N, T = 512, 2048, 6
    eager, graphed = _layer(env, D, N, B, period), _layer(env, D, N, B, period)
    sc = synth.dim_scales(0, D)
    X = up(env, synth.prompt(0, 32, sc))
    for f in (eager, graphed):
        f.prefill_partition(X)
    xs = [up(env, synth.decode_input(0, t, B, sc)) for t in range(T)]
    y_eager = [eager.decode_step(x).clone() for x in xs]
    ys = [torch.empty((B, D), dtype=torch.float32, device=dev) for _ in range(T)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for x, y in zip(xs, ys):
            graphed.decode_step(x, y)
    assert graphed.step_count() == 0  # capturing runs nothing
    g.replay()
    torch.cuda.synchronize()
    for t in range(T):
        assert torch.equal(ys[t], y_eager[t]), f"step {t}"
    assert graphed.step_count() == T
    assert np.array_equal(graphed.selected(), eager.selected())
    graphed.check()
    eager.check()
    eager.close()
    graphed.close()


def test_moe_decode_steps_replay_from_a_graph(env):
    pop, torch, dev = env
    E, D, N, B, T = 4, 256, 1024, 8, 4
    ws = [synth.ffn_weights(0, D, N, layer=e) for e in range(E)]

    def moe():
        return pop.PopMoE([up(env, w[0]) for w in ws], [up(env, w[1]) for w in ws], [up(env, w[2]) for w in ws],
                          r=0.3, gamma=0.1, max_batch=B, max_prefill_tokens=64)
    eager, graphed = moe(), moe()
    sc = synth.dim_scales(0, D)
    X = up(env, synth.prompt(0, 48, sc))
    L = torch.from_numpy(synth.router_logits(0, 48, E).astype(np.float32)).to(dev)
    for m in (eager, graphed):
        m.prefill_partition(X, L)
    xs = [up(env, synth.decode_input(0, t, B, sc)) for t in range(T)]
    ls = [torch.from_numpy(synth.router_logits(0, B, E, step=t).astype(np.float32)).to(dev) for t in range(T)]
    y_eager = [eager.decode_step(x, l).clone() for x, l in zip(xs, ls)]
    ys = [torch.empty((B, D), dtype=torch.float32, device=dev) for _ in range(T)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for x, l, y in zip(xs, ls, ys):
            graphed.decode_step(x, l, y)
    g.replay()
    torch.cuda.synchronize()
    for t in range(T):
        assert torch.equal(ys[t], y_eager[t]), f"step {t}"
    graphed.check()
    eager.close()
    graphed.close()
