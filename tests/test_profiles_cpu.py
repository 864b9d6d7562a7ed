"""Structural checks of the committed ncu summaries (profiles/*.md), no GPU
needed: the counters recorded there must match what the kernels are meant to
do.

- Causal prefill: the tensor pipe's active cycles equal the MMA work of the
  lower-triangle tile count (no tile past the diagonal is computed, none twice).
- Decode: DRAM bytes read equal the K/V bytes once, whether the 8 query heads of
  a KV head (plain decode) or 64 query rows (multi-token decode on the tensor
  cores) share them, and whether the cache is contiguous or in shuffled pages:
  the reads do not grow with G, with the rows or with the page gather.
"""
import os
import re

import pytest

PROFILES = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles")
KV_BYTES_32K = 2 * 32768 * 8 * 128 * 2          # Llama3-70B, B = 1, ctx 32768, bf16
FP8_BYTES_32K = 2 * 32768 * (8 * 128 + 4)       # E4M3 codes + one fp32 scale per token
UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}


def _read(name):
    path = os.path.join(PROFILES, name)
    if not os.path.exists(path):
        pytest.skip(f"{name} not captured")
    return open(path).read()


def _dram_read(text):
    m = re.search(r"DRAM read \(`dram__bytes_read\.sum`\) \| ([0-9.]+) (\w+) \|", text)
    assert m, "no DRAM read line"
    return float(m.group(1)) * UNITS[m.group(2)]


def test_prefill_tensor_work_is_the_causal_tile_count():
    text = _read("prefill_causal_llama70b_s8192.md")
    m = re.search(r"- ratio ([0-9.]+)", text)
    assert m, "no structural check in the prefill summary"
    assert abs(float(m.group(1)) - 1.0) < 0.01
    # and the expected MMA count is the one of 8K causal tiles: 32 (KV head,
    # head pair) items per query tile, sum over query tiles of (qt + 1) key
    # tiles, 2 heads x (8 S + 8 P V) instructions per key tile
    n_qt = 8192 // 128
    assert f"expected: {32 * n_qt * (n_qt + 1) // 2 * 32} MMAs" in text


@pytest.mark.parametrize("name,algo", [
    ("decode_split_llama70b_ctx32768.md", KV_BYTES_32K),        # 8 query heads per KV head
    ("decode_tc_multi8_llama70b_ctx32768.md", KV_BYTES_32K),    # 64 query rows per KV head
    ("decode_fp8_llama70b_ctx32768.md", FP8_BYTES_32K),
    ("decode_paged16_llama70b_ctx32768.md", KV_BYTES_32K),     # 2048 shuffled 16-token pages
])
def test_decode_reads_the_cache_once(name, algo):
    read = _dram_read(_read(name))
    assert 0.99 * algo <= read <= 1.05 * algo, (read, algo)
