"""The C-ABI library without a GPU: it loads, exports every symbol include/*.h declares,
and its host-side logic (region counts, argument checks) agrees with the oracle."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pop():
    import __graft_entry__
    __graft_entry__.build()
    import online_structured_ffn_gb300 as pop
    return pop


def _declared_functions():
    inc = os.path.join(ROOT, "include")
    text = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pop_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(pop):
    names = _declared_functions()
    assert len(names) >= 18
    lib = ctypes.CDLL(pop.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) == set(pop.SIGNATURES), "binding and header disagree"


def test_build_targets_sm103a_only(pop, monkeypatch):
    """Every nvcc command of the build (compile and link) names exactly one target, sm_103a, and
    the library lands in-tree. The commands are intercepted, not run."""
    import importlib.util
    import subprocess
    spec = importlib.util.spec_from_file_location("_pop_build_t", os.path.join(ROOT, "online_structured_ffn_gb300",
                                                                              "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    cmds = []

    class Done:
        returncode, stdout, stderr = 0, "", ""

    def fake_run(cmd, **kw):
        cmds.append(list(cmd))
        out = cmd[cmd.index("-o") + 1]
        open(out, "wb").close()  # stands in for the object or library nvcc would write
        return Done()

    monkeypatch.setattr(subprocess, "run", fake_run)
    monkeypatch.setattr(b, "LIB", os.path.join(ROOT, "_pytest_fake_lib.so"))
    monkeypatch.setattr(b, "BUILD_DIR", os.path.join(ROOT, "_pytest_fake_build"))
    try:
        b.build(force=True)
    finally:
        import shutil
        shutil.rmtree(os.path.join(ROOT, "_pytest_fake_build"), ignore_errors=True)
        if os.path.exists(os.path.join(ROOT, "_pytest_fake_lib.so")):
            os.remove(os.path.join(ROOT, "_pytest_fake_lib.so"))
    assert len(cmds) == len(b.sources()) + 1  # one compile per .cu file, one link
    for c in cmds:
        targets = [c[i + 1] for i, a in enumerate(c) if a in ("-gencode", "-arch", "--gpu-architecture")]
        targets += [a for a in c if a.startswith(("-arch=", "--gpu-architecture=", "-gencode="))]
        assert targets == ["arch=compute_103a,code=sm_103a"], c
    assert os.path.dirname(pop.LIB_PATH).endswith("online_structured_ffn_gb300")


@pytest.mark.parametrize("N", [0, 1, 7, 100, 1000, 1024, 11008, 14336, 28672, 49152])
@pytest.mark.parametrize("r,gamma", [(0.3, 0.1), (0.299, 0.1), (0.5, 0.1), (0.0, 0.1), (0.3, 0.0), (0.4, 0.6),
                                     (1.0, 0.1), (0.25, 0.05), (0.125, 0.125)])
def test_region_counts_match_oracle(pop, N, r, gamma):
    ref = oracle.region_counts(N, r, gamma)
    got = pop.pop_region_counts(N, r, gamma)
    assert (got.n_P, got.n_R, got.n_C, got.keep, got.k) == (ref.n_P, ref.n_R, ref.n_C, ref.keep, ref.k)


def test_region_counts_rejects_bad_args(pop):
    for N, r, g in [(10, -0.1, 0.1), (10, 1.1, 0.1), (10, 0.3, -0.5), (-1, 0.3, 0.1)]:
        with pytest.raises(pop.PopError) as e:
            pop.pop_region_counts(N, r, g)
        assert e.value.status == pop.POP_ERR_INVALID_ARG
    assert pop.load_library().pop_region_counts(10, 0.3, 0.1, None) == pop.POP_ERR_INVALID_ARG


def test_create_rejects_bad_config_before_touching_cuda(pop):
    lib = pop.load_library()
    out = ctypes.c_void_p(1)
    good = dict(D=256, D_FF=1024, r=0.3, gamma=0.1, period=1, max_batch=1, max_prefill_tokens=64, out_f32=1)
    fake = 4096  # any 16-byte aligned non-null value: the checks below fail before it is used
    bad = [dict(D=100), dict(D=0), dict(D=20000), dict(D_FF=0), dict(D_FF=60000), dict(period=0),
           dict(max_batch=0), dict(max_batch=65), dict(max_prefill_tokens=0), dict(r=1.5), dict(gamma=-1.0),
           dict(skip=2), dict(skip=-1)]
    for b in bad:
        cfg = pop.pop_config(**{**good, **b})
        assert lib.pop_ffn_create(ctypes.byref(cfg), fake, fake, fake, None, ctypes.byref(out)) == \
            pop.POP_ERR_INVALID_ARG, b
        assert out.value is None
        assert lib.pop_last_error(None)
    cfg = pop.pop_config(**good)
    assert lib.pop_ffn_create(ctypes.byref(cfg), None, fake, fake, None, ctypes.byref(out)) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_ffn_create(ctypes.byref(cfg), fake + 2, fake, fake, None, ctypes.byref(out)) == \
        pop.POP_ERR_INVALID_ARG  # misaligned
    assert lib.pop_ffn_create(None, fake, fake, fake, None, ctypes.byref(out)) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_ffn_create(ctypes.byref(cfg), fake, fake, fake, None, None) == pop.POP_ERR_INVALID_ARG


def test_null_handle_calls(pop):
    lib = pop.load_library()
    assert lib.pop_prefill_partition(None, 4096, 1, None, None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_decode_step(None, 4096, 1, 4096, None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_ffn_dense_ref(None, 4096, 1, 4096, None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_check(None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_set_wait_limit(None, 5) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_get_partition(None, None, None, None) == pop.POP_ERR_INVALID_ARG
    assert b"NULL" in lib.pop_last_error(None)
    lib.pop_ffn_destroy(None)  # no-op


def test_status_strings(pop):
    lib = pop.load_library()
    for s in range(8):
        assert lib.pop_status_string(s).decode() == pop.status_name(s)
    assert lib.pop_status_string(99) == b"POP_ERR_UNKNOWN"


def test_moe_rejects_bad_arguments_before_touching_cuda(pop):
    lib = pop.load_library()
    out = ctypes.c_void_p(1)
    fake = 4096
    good = dict(D=256, D_FF=1024, r=0.3, gamma=0.1, period=1, max_batch=4, max_prefill_tokens=64, out_f32=1)
    cfg = pop.pop_config(**good)

    def ptrs(n, v=fake):
        return (ctypes.c_void_p * n)(*([v] * n))

    for E in (0, 1, 257):
        n = max(E, 1)
        assert lib.pop_moe_create(ctypes.byref(cfg), E, ptrs(n), ptrs(n), ptrs(n), None, ctypes.byref(out)) == \
            pop.POP_ERR_INVALID_ARG
        assert out.value is None
    assert lib.pop_moe_create(ctypes.byref(cfg), 2, None, ptrs(2), ptrs(2), None, ctypes.byref(out)) == \
        pop.POP_ERR_INVALID_ARG
    holes = (ctypes.c_void_p * 2)(fake, None)
    assert lib.pop_moe_create(ctypes.byref(cfg), 2, ptrs(2), holes, ptrs(2), None, ctypes.byref(out)) == \
        pop.POP_ERR_INVALID_ARG
    bad = pop.pop_config(**{**good, "D": 100})  # rejected by the first expert's create, before CUDA
    assert lib.pop_moe_create(ctypes.byref(bad), 2, ptrs(2), ptrs(2), ptrs(2), None, ctypes.byref(out)) == \
        pop.POP_ERR_INVALID_ARG
    assert b"expert 0" in lib.pop_moe_last_error(None)
    assert lib.pop_moe_create(ctypes.byref(cfg), 2, ptrs(2), ptrs(2), ptrs(2), None, None) == pop.POP_ERR_INVALID_ARG
    # NULL handles
    assert lib.pop_moe_prefill_partition(None, fake, fake, 1, None, None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_moe_decode_step(None, fake, fake, 1, fake, None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_moe_check(None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_moe_get_counts(None, None) == pop.POP_ERR_INVALID_ARG
    T = ctypes.c_int(0)
    assert lib.pop_moe_get_routing(None, ctypes.byref(T), None, None) == pop.POP_ERR_INVALID_ARG
    assert lib.pop_moe_expert(None, 0) is None
    assert lib.pop_moe_num_experts(None) == -1
    assert lib.pop_moe_set_concurrent(None, 1) == pop.POP_ERR_INVALID_ARG
    lib.pop_moe_destroy(None)  # no-op


def test_binding_checks_tensor_arguments_before_the_c_abi(pop):
    # the wrappers check dtype, contiguity and shape on the host; nothing reaches the library
    torch = pytest.importorskip("torch")
    f = pop.PopFFN.__new__(pop.PopFFN)
    f.handle, f.D, f.N = None, 8, 16
    f.cfg = pop.pop_config(D=8, D_FF=16, r=0.3, gamma=0.1, period=1, max_batch=4, max_prefill_tokens=8, out_f32=1)
    good_x = torch.zeros((2, 8), dtype=torch.bfloat16)
    for bad in (torch.zeros((2, 8), dtype=torch.float32), torch.zeros((2, 9), dtype=torch.bfloat16),
                torch.zeros((8, 2), dtype=torch.bfloat16).t(), torch.zeros(8, dtype=torch.bfloat16)):
        with pytest.raises(pop.PopError) as e:
            f.decode_step(bad)
        assert e.value.status == pop.POP_ERR_INVALID_ARG
    with pytest.raises(pop.PopError):
        f.decode_step(good_x, torch.zeros((2, 8), dtype=torch.bfloat16))  # y of the wrong dtype
    with pytest.raises(pop.PopError):
        f.partition_from_importance(torch.zeros(15, dtype=torch.float32))
    m = pop.PopMoE.__new__(pop.PopMoE)
    m.handle, m.D, m.N, m.E, m.cfg = None, 8, 16, 4, f.cfg
    with pytest.raises(pop.PopError):
        m.decode_step(good_x, torch.zeros((2, 4), dtype=torch.float64))  # logits must be float32
    with pytest.raises(pop.PopError):
        m.prefill_partition(good_x, torch.zeros((1, 4), dtype=torch.float32))  # a row per token
    with pytest.raises(pop.PopError):
        f.decode_step(good_x, torch.zeros((1, 8), dtype=torch.float32))  # y too short
