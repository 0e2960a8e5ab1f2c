"""Host-side logic of bench.py without a GPU: the algorithmic byte counts behind the roofline, the
launch counts it reports, and the code hash that ties a committed ncu summary to the kernels it
measured."""
import os
import types

import pytest

import bench
import oracle


def _counts(N, r, gamma):
    c = oracle.region_counts(N, r, gamma)
    return types.SimpleNamespace(n_R=c.n_R, n_C=c.n_C, n_P=c.n_P, keep=c.keep, k=c.k)


def test_touched_bytes_of_the_7b_workloads():
    # gate/up rows of R u C and down columns of R u S, bf16
    c = _counts(11008, 0.299, 0.1)
    gu, dn = bench.touched_bytes(c, 4096)
    assert gu == 2 * (6616 + 2201) * 4096 * 2 and dn == 7717 * 4096 * 2
    assert (gu + dn) / 1e6 == pytest.approx(207.675392)


def test_touched_bytes_of_the_skip_variant_average_over_a_period():
    c = _counts(28672, 0.5, 0.1)
    P = 16
    full, dn = bench.touched_bytes(c, 8192)
    skip, dn2 = bench.touched_bytes(c, 8192, dict(skip=True, period=P))
    assert dn2 == dn
    rows = ((c.n_R + c.n_C) + (P - 1) * (c.n_R + c.k)) / P
    assert skip == pytest.approx(2 * rows * 8192 * 2)
    assert skip < full
    # period 1: every step is an update
    assert bench.touched_bytes(c, 8192, dict(skip=True, period=1))[0] == full


def _stack(wl, counts, chunks):
    return types.SimpleNamespace(wl=wl, counts=counts, chunks=chunks)


def test_launch_counts_per_session():
    b1 = dict(bench.WORKLOADS["llama2-7b-ffn-b1"])
    c1 = _counts(b1["N"], b1["r"], b1["gamma"])
    n1 = bench.Stack.launches_per_session(_stack(b1, c1, 1))
    assert n1 == b1["layers"] * ((3 + 1) + 2 * b1["T"])  # prefill: 3 per chunk + partition
    b16 = dict(bench.WORKLOADS["llama2-7b-ffn-b16"])
    c16 = _counts(b16["N"], b16["r"], b16["gamma"])
    n16 = bench.Stack.launches_per_session(_stack(b16, c16, 4))
    assert n16 == b16["layers"] * ((3 * 4 + 1 + 2) + 2 * b16["T"])  # + the two slab builders
    fd = dict(bench.WORKLOADS["llama2-7b-ffn-b1-fulldyn"])
    cfd = _counts(fd["N"], fd["r"], fd["gamma"])
    assert cfd.n_C > 8192  # the separate top-k kernel runs every step
    assert bench.Stack.launches_per_session(_stack(fd, cfd, 1)) == fd["layers"] * (4 + 3 * fd["T"])
    sk = dict(bench.WORKLOADS["llama-70b-ffn-b64-p16-skip"])
    csk = _counts(sk["N"], sk["r"], sk["gamma"])
    updates = (sk["T"] + sk["period"] - 1) // sk["period"]
    chunks = (sk["M"] + sk["chunk"] - 1) // sk["chunk"]
    assert bench.Stack.launches_per_session(_stack(sk, csk, chunks)) == \
        sk["layers"] * ((3 * chunks + 1 + 2) + 2 * sk["T"] + updates)


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text("int f() {\n  return 1;  // one\n}\n")
    b.write_text("/* a block\n   comment */\nint f() {\n\n  return 1;\n}\n// trailing\n")
    c.write_text("int f() {\n  return 2;\n}\n")
    assert bench.code_hash(str(a)) == bench.code_hash(str(b))
    assert bench.code_hash(str(a)) != bench.code_hash(str(c))


def test_traffic_is_read_only_for_the_code_it_was_measured_on(monkeypatch):
    path = os.path.join(bench.ROOT, "profiles", "gateup_decode_llama2-7b-ffn-b1.md")
    text = open(path).read()
    recorded = [ln.split("`")[1] for ln in text.splitlines() if "source_sha256_16" in ln][0]
    monkeypatch.setattr(bench, "code_hash", lambda p: recorded)
    assert bench.traffic_from_profiles("gateup_decode", "llama2-7b-ffn-b1") > 1e8
    monkeypatch.setattr(bench, "code_hash", lambda p: "0" * 16)
    assert bench.traffic_from_profiles("gateup_decode", "llama2-7b-ffn-b1") is None
    assert bench.traffic_from_profiles("gateup_decode", "no-such-workload") is None
