"""Host-side launch logic of the attention kernels, compiled from the library's own header
with the host compiler: the rule that decides when the forward and the dQ kernel deal
their work items in two groups of slices (so that each group's K and V stay in L2)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <cstdio>
#include "kernels.h"
int main() {
  const long long MiB = 1ll << 20;
  const struct { int n; long long bytes; } cases[] = {
      {16, 4 * MiB}, {16, 2 * MiB}, {15, 4 * MiB}, {10, 4 * MiB}, {12, 4 * MiB},
      {6, 8 * MiB}, {1, 64 * MiB}, {2, 64 * MiB}, {64, MiB / 2}, {128, MiB / 2}};
  for (const auto& c : cases) printf("%d\n", attn::slices_per_group(c.n, c.bytes));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.isdir(CUDA_INC), reason="needs g++ and the CUDA headers")
def test_slices_per_group_rule(tmp_path):
    """Two groups of half the slices exactly when the slices' re-read bytes exceed 40 MiB
    and the slice count is even; otherwise one group. long8k at d = 128 (16 slices of
    4 MiB of K and V) splits into two groups of eight; gpt205m at d = 64 (64 slices of
    0.5 MiB) stays one group."""
    src = tmp_path / "spg.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "spg"
    subprocess.run(["g++", "-std=c++17", "-I", os.path.join(ROOT, "causal_attention_gb300", "csrc"), "-I", CUDA_INC,
                    str(src), "-o", str(exe)], check=True, capture_output=True, timeout=120)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    # 64 MiB > 40 -> 8; 32 MiB -> all; odd count -> all; exactly 40 MiB -> all; 48 -> 6;
    # 48 -> 3 (odd groups are fine); a single slice -> 1; 128 MiB over 2 slices -> 1;
    # 32 MiB -> all; 64 MiB over 128 slices -> 64
    assert got == [8, 16, 15, 10, 6, 3, 1, 1, 64, 64]
