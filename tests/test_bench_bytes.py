"""The roofline's numerator: bench.attention_bytes against the per-launch
bytes written out by hand for the headline workload (32 requests of 8192
context tokens, 64 query / 8 kv heads, D = 128, 16-token pages): e4m3 K and V
of every context token (2 x 8 x 128 bytes), one 4-byte page-table entry per
16 tokens, bf16 queries, fp32 outputs and log-sum-exps."""
import bench
from workloads import b32_8k


def test_b32_8k_bytes_by_hand():
    wl = b32_8k()
    tokens = 32 * 8192
    kv_fp8 = tokens * 2 * 8 * 128
    table = 32 * (8192 // 16) * 4
    q = 32 * 64 * 128 * 2
    out = 32 * 64 * 128 * 4 + 32 * 64 * 4
    assert bench.attention_bytes(wl, 0, True) == kv_fp8 + table + q + out == 538_517_504
    assert bench.attention_bytes(wl, 0, False) == 2 * kv_fp8 + table + q + out == 1_075_388_416

