"""The folded-readout kernel's shared-memory work areas (host arithmetic, no GPU): the sizes that decide how many
units an SM holds at once. A unit of the int4 symmetric state and of the buffered bf16 state must fit sixteen to
an SM (the batch-64, 32-head launch then runs in one wave of 2,048 units), one with 32-token tables six (the
768 units of the long-context shape in one wave). Compiled with nvcc for the host; skipped without it."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_gated_delta_gb300", "csrc")
SMEM_PER_SM = 233472          # bytes of shared memory an SM gives its blocks
RESERVED = 1024               # bytes the hardware keeps per block

PROBE = r'''
#include "decode_fold.cuh"
#include <cstdio>
int main() {
  const int cfg[][6] = {{128, 64, 0, 0, 0, 8}, {128, 64, 0, 0, 1, 8}, {128, 64, 0, 0, 0, 32}, {128, 32, 1, 1, 0, 8},
                        {64, 64, 0, 0, 0, 8}, {64, 64, 0, 0, 0, 32}};
  for (const auto &c : cfg) {
    const pace::FoldSmem L = pace::fold_smem(c[0], c[1], c[2], c[3], c[4], c[5]);
    std::printf("%d %d %d %d %d %d %zu %zu %zu %zu %zu\n", c[0], c[1], c[2], c[3], c[4], c[5], L.total, L.pb, L.kbf,
                L.vrow, L.gram);
  }
  return 0;
}
'''


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    return None


@pytest.fixture(scope="module")
def layouts():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "probe.cu")
        exe = os.path.join(tmp, "probe")
        with open(src, "w") as f:
            f.write(PROBE)
        r = subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC, "-I",
                            os.path.join(ROOT, "include"), src, "-o", exe], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    res = {}
    for line in out.split("\n"):
        if line.strip():
            v = [int(x) for x in line.split()]
            res[tuple(v[:6])] = dict(total=v[6], pb=v[7], kbf=v[8], vrow=v[9], gram=v[10])
    return res


def units_per_sm(total):
    return SMEM_PER_SM // (total + RESERVED)


def test_int4_symmetric_unit_fits_sixteen_per_sm(layouts):
    assert units_per_sm(layouts[(128, 64, 0, 0, 0, 8)]["total"]) >= 16


def test_buffered_bf16_unit_fits_sixteen_per_sm(layouts):
    assert units_per_sm(layouts[(128, 64, 0, 0, 1, 8)]["total"]) >= 16


def test_32_token_tables_fit_six_per_sm(layouts):
    assert units_per_sm(layouts[(128, 64, 0, 0, 0, 32)]["total"]) >= 6


def test_staged_code_words_fit_their_area(layouts):
    """Steps without a rounding stage the unit's int4 code words (d*d/2 bytes) from pb onwards: the area from pb
    to the end of the work area must hold them."""
    for key, L in layouts.items():
        d, bf = key[0], key[4]
        if not bf:
            assert L["total"] - L["pb"] >= d * d // 2, key


def test_32_token_key_table_fits_over_values_and_gram(layouts):
    """With 32-token tables the rounding's fp16 key table (d x 16 pairs) is built over the value rows and the
    Gram/L area, which must be contiguous and large enough."""
    for key, L in layouts.items():
        if key[5] == 32:
            d = key[0]
            assert L["kbf"] == L["vrow"]
            assert L["gram"] >= L["vrow"] + 32 * d          # the Gram area follows the value rows
            assert L["gram"] + 32 * 32 * 4 - L["kbf"] >= d * 16 * 4, key
