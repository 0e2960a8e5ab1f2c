"""The allocation-free dense single-token entry point, called through the C ABI.

Some callers cannot allocate GPU memory while they run (their device memory is reserved up
front by their own memory manager, or their loop must not enter the CUDA allocator), so
pop_ffn_dense_token_noalloc keeps its scratch in a static device array instead. Its output must
agree with the handle-based dense path (pop_ffn_dense_ref) on the same weights, and with the CPU
oracle's dense FFN, on two calls in a row that share that array. This file is collected last on
purpose.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import online_structured_ffn_gb300 as pop
    torch.cuda.set_device(0)
    return pop, torch, torch.device("cuda", 0)


def _up(torch, dev, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


@pytest.mark.parametrize("D,N,out_f32", [(4096, 11008, 1), (512, 2048, 1), (264, 1000, 0)])
def test_noalloc_matches_dense_ref_twice(env, D, N, out_f32):
    pop, torch, dev = env
    lib = pop.load_library()
    Wg, W1, W2 = synth.ffn_weights(5, D, N)
    sc = synth.dim_scales(5, D)
    g, u, w = _up(torch, dev, Wg), _up(torch, dev, W1), _up(torch, dev, W2)
    ref = pop.PopFFN(g, u, w, r=0.3, gamma=0.1, max_batch=1, max_prefill_tokens=16, out_f32=bool(out_f32))
    ydt = torch.float32 if out_f32 else torch.bfloat16
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):
        x = _up(torch, dev, synth.decode_input(5, step, 1, sc))
        y = torch.full((1, D), float("nan"), dtype=ydt, device=dev)
        st = lib.pop_ffn_dense_token_noalloc(g.data_ptr(), u.data_ptr(), w.data_ptr(), D, N, x.data_ptr(),
                                             y.data_ptr(), out_f32, stream)
        assert st == pop.POP_OK, lib.pop_last_error(None)
        y_ref = ref.dense_ref(x)
        torch.cuda.synchronize()
        a, b = y.float().cpu().numpy(), y_ref.float().cpu().numpy()
        assert np.all(np.isfinite(a))
        parity.check_y(a, b, f"no-alloc call {step} against pop_ffn_dense_ref")
        f64 = synth.bf16_to_f64
        y_or = oracle.dense_ffn(f64(Wg), f64(W1), f64(W2), f64(synth.decode_input(5, step, 1, sc)))
        parity.check_y(a, y_or, f"no-alloc call {step} against the oracle")
    ref.close()


def test_noalloc_rejects_sizes_beyond_its_scratch(env):
    pop, torch, dev = env
    lib = pop.load_library()
    buf = torch.zeros(64, dtype=torch.float32, device=dev)
    p = buf.data_ptr()
    too_big = pop.POP_STATIC_MAX_D_FF + 8
    assert lib.pop_ffn_dense_token_noalloc(p, p, p, 64, too_big, p, p, 1, None) == pop.POP_ERR_INVALID_ARG
    assert b"POP_STATIC_MAX_D_FF" in lib.pop_last_error(None)
    assert lib.pop_ffn_dense_token_noalloc(p, p, p, 60, 64, p, p, 1, None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_ffn_dense_token_noalloc(None, p, p, 64, 64, p, p, 1, None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_ffn_dense_token_noalloc(p + 4, p, p, 64, 64, p, p, 1, None) == pop.POP_ERR_INVALID_ARG
