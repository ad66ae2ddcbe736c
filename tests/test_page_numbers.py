"""The byte/bandwidth accounting reproduces the kernel table the pages print,
and the head-size arithmetic the pages state."""
import math

from conftest import read_kv
from draft_vocab_lm_gb300 import roofline


def test_effective_bandwidth_rows_of_the_kernel_table():
    p = read_kv("page_numbers.txt")
    spec = float(p["gb10_GBs"])
    for pre in ("lm_head", "gdn"):
        rows, K = int(p[pre + "_rows"]), int(p[pre + "_K"])
        mb = roofline.head_bytes(rows, K, "bf16") / 1e6
        assert round(mb, 1) == float(p[pre + "_MB"])
        # the table divides the rounded megabytes by the time
        gbs = roofline.effective_gbs(float(p[pre + "_MB"]) * 1e6, int(p[pre + "_us"]) * 1e-6)
        assert math.floor(gbs) == int(p[pre + "_GBs"])
        assert round(100 * int(p[pre + "_GBs"]) / spec) == int(p[pre + "_pct"])


def test_head_split_and_trim_ratio():
    p = read_kv("page_numbers.txt")
    assert int(p["vocab"]) // int(p["tp"]) == int(p["lm_head_rows"])
    assert round(int(p["vocab"]) / int(p["trim_rows"]), 1) == float(p["trim_ratio"])
    # the trimmed head's read shrinks by exactly the row ratio
    full = roofline.head_bytes(int(p["vocab"]), 5120)
    trim = roofline.head_bytes(int(p["trim_rows"]), 5120)
    assert round(full / trim, 1) == float(p["trim_ratio"])


def test_call_bytes_of_the_workloads():
    # bf16 shortlist 16,000 x 2,560 at M=1: head + hidden + one result
    assert roofline.call_bytes(16000, 2560, 1) == 81_920_000 + 5_120 + 12
    assert roofline.head_bytes(248_320, 2560) == 1_271_398_400
    assert roofline.head_bytes(32768, 5120, "nvfp4") == 83_886_080 + 10_485_760 + 4
    assert roofline.trim_bytes(32768, 10240) == 2 * 335_544_320 + 131_072
