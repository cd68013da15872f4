"""Host-side pieces of bench.py that need no GPU: the work counts the
roofline divides by, and the rule that the committed DRAM traffic is
reported only for the kernel sources it was measured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_step_flops_and_gemm_bytes():
    T = 8192
    shapes = [(4096, 12288), (4096, 4096), (4096, 16384), (16384, 4096)]
    flops = sum(3 * 2 * T * a * b for a, b in shapes)
    assert bench.step_flops() == flops
    assert abs(flops / 1e9 - 9895.6) < 0.1
    b = bench.gemm_algorithmic_bytes()
    assert len(b) == 12
    # fprop of FC2: X 8192x16384, W 4096x16384 (1 B each), Y 8192x4096 bf16
    assert b[9] == 8192 * 16384 + 4096 * 16384 + 2 * 8192 * 4096
    # wgrad of QKV: dY^T 12288x8192, X^T 4096x8192, dW 12288x4096 bf16
    assert b[2] == 12288 * 8192 + 4096 * 8192 + 2 * 12288 * 4096


def test_traffic_only_for_the_profiled_sources(monkeypatch):
    import re

    text = open(bench.GEMM_PROFILE).read()
    want = int(re.search(r"^gemm_traffic_bytes_per_launch: (\d+)$", text, re.M).group(1))
    sha = re.search(r"^gemm_source_sha256: ([0-9a-f]{64})$", text, re.M).group(1)
    monkeypatch.setattr(bench, "gemm_source_sha256", lambda: sha)
    assert bench.gemm_traffic() == want
    monkeypatch.setattr(bench, "gemm_source_sha256", lambda: "0" * 64)
    assert bench.gemm_traffic() is None
    alg = int(re.search(r"^gemm_algorithmic_bytes_per_launch: (\d+)$", text, re.M).group(1))
    assert alg == sum(bench.gemm_algorithmic_bytes()) // 12


def test_source_hash_is_sha256_of_the_kernel_files():
    import hashlib

    h = hashlib.sha256()
    for name in bench.GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, "fp8_mixed_precision_history_gb300", "csrc", name), "rb").read())
    assert bench.gemm_source_sha256() == h.hexdigest()


def test_cast_bytes_per_step():
    """3 B per element (bf16 read + FP8 codes written) for the casts of X, W and
    dY of the four layers; 4 B with transposed copies."""
    import bench

    T = 8192
    elements = sum(T * fin + fout * fin + T * fout for _, fin, fout in bench.layers())
    assert elements == 738197504
    assert bench.cast_bytes() == 3 * elements
    assert bench.cast_bytes(transposed=True) == 4 * elements
    assert bench.step_flops() == 9895604649984


def test_oracle_sample_size_shrinks_below_the_fixed_cost():
    """The reference arm's samples: a budget below the 8-token step's cost
    divides every layer's output features by a power of two, and the sample
    then does the matching share of the step's work."""
    tokens, div = bench.oracle_sample_size(1e-3)
    assert tokens == 8 and div >= 2 and div & (div - 1) == 0 and div <= 256
    flop, sec = bench.oracle_step_sample(tokens, div)
    fo = [max(16, fout // div) for _, _, fout in bench.layers()]
    assert flop == sum(3 * 2 * tokens * fin * f for (_, fin, _), f in zip(bench.layers(), fo))
    assert sec > 0
    assert "output features / %d" % div in bench.sample_text(tokens, div)


def test_oracle_thread_count_follows_the_setter():
    """The bench's oracle legs set the oracle's threads to every host core, so
    a launcher's OMP_NUM_THREADS=1 does not leave rank 0 on one core."""
    import oracle

    before = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        assert oracle.num_threads() == 1
        oracle.set_num_threads(bench.cpu_cores())
        assert oracle.num_threads() == bench.cpu_cores()
    finally:
        oracle.set_num_threads(before)
