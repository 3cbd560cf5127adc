"""The benchmark's roofline numerator is the oracle's byte count: bench.kv_bytes, the
algorithmic bytes per step that the roofline divides by the kernel time, must equal the
oracle's decode_bytes (pinned to the cost model's KV term in test_oracle_pins) term by term
on every workload's sequence lengths, for block top-k and for dense decode."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle as O  # noqa: E402
import workloads as W  # noqa: E402


@pytest.mark.parametrize("cfg", W.CONFIGS, ids=lambda c: c.name)
def test_roofline_bytes_are_the_oracle_byte_count(cfg):
    lens = [int(x) for x in W._draw_lengths(cfg)]
    es = 2 if cfg.dtype == "bf16" else 4
    got = bench.kv_bytes(cfg, lens)
    want = O.decode_bytes(lens, cfg.num_kv_heads, cfg.group, cfg.head_dim, cfg.top_k, es)
    assert got["kv"] == want["kv"]
    assert got["centroids"] == want["centroids"]
    assert got["qo"] == want["qo"]
    dense = O.decode_bytes(lens, cfg.num_kv_heads, cfg.group, cfg.head_dim, None, es)
    assert got["dense_kv"] == dense["kv"]


def test_config1_step_bytes():
    # Qwen3-0.6B-shaped workload: 64 x 8 rows, 63 full pages + the final page of 16 tokens
    # kept per row, 511 scored centroids per row, q and out of 64 x 16 heads; plus the 64 x 8
    # appended centroids of the pages the current token completed (context 8192 = 512 full
    # pages): 336,068,608 bytes, the figure the roofline uses.
    cfg = W.find_config("qwen3-0.6b")
    byt = bench.kv_bytes(cfg, [8192] * 64)
    append = 64 * 8 * 128 * 2
    assert byt["kv"] == 64 * 8 * 64 * 16 * 128 * 2 * 2
    assert byt["centroids"] == 64 * 8 * 511 * 128 * 2
    assert byt["kv"] + byt["centroids"] + byt["qo"] + append == 336068608


def test_kernel_fingerprint_ignores_comments_only():
    # the traffic record stays valid across comment edits and goes stale on code edits
    code = 'int f(int x) { return x + 1; }  // adds one\n/* block */ const char *s = "a//b";\n'
    same = '// header\nint f(int x)   {\n  return x + 1;   /* body */ }\nconst char *s = "a//b";\n'
    other = 'int f(int x) { return x + 2; }\nconst char *s = "a//b";\n'
    strip = bench.strip_comments
    assert strip(code) == strip(same)
    assert strip(code) != strip(other)
    assert '"a//b"' in strip(code)                        # string literals are kept whole
    files = {f: code for f in bench.KERNEL_SOURCES}
    fp = bench.kernel_source_sha(files.get)
    assert bench.kernel_source_sha({f: same for f in bench.KERNEL_SOURCES}.get) == fp
    assert bench.kernel_source_sha({f: other for f in bench.KERNEL_SOURCES}.get) != fp
