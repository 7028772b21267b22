"""The debug-checks build's address predicates (csrc/checks.h), pinned on the host.

The header is plain C++, so a small program compiled with g++ exercises each
predicate on both sides of its boundary: a 16-byte aligned TMA x against one off
by an element, a store at coordinate 0 against -1, the last TMEM column against
one past it, the warp's own TMEM quadrant against its neighbour, and the N field
of the instruction descriptor the kernels build. No GPU involved."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "alibi_positional_bias_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "checks.h"
using namespace alibi::check;
static int fails = 0;
#define EXPECT(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); ++fails; } } while (0)
int main()
{
    // TMA x of 16-bit elements: multiples of 8 (16 bytes)
    EXPECT(tma_x_aligned(0) && tma_x_aligned(64) && tma_x_aligned(-8));
    EXPECT(!tma_x_aligned(1) && !tma_x_aligned(7) && !tma_x_aligned(60));
    // stores: aligned x and no negative coordinate
    EXPECT(tma_store_coords(32, 0, 0) && tma_store_coords(0, 127, 5));
    EXPECT(!tma_store_coords(-8, 0, 0) && !tma_store_coords(0, -1, 0) && !tma_store_coords(0, 0, -1));
    EXPECT(!tma_store_coords(4, 0, 0));
    // shared-memory window [1024, 1024 + 4096), 16 KB box needs the whole box inside
    EXPECT(smem_range(1024, 4096, 1024, 1024, 5120));
    EXPECT(!smem_range(1024, 4097, 1024, 1024, 5120));
    EXPECT(!smem_range(2048 + 16, 16, 1024, 1024, 5120));   // misaligned for a 1024-byte atom
    EXPECT(smem_range(2048 + 16, 16, 16, 1024, 5120));
    EXPECT(!smem_range(1008, 16, 16, 1024, 5120));           // below the window
    EXPECT(!smem_range(5120, 16, 16, 1024, 5120));           // at its end
    EXPECT(!smem_range(0xFFFFFFF0u, 32, 16, 1024, 0xFFFFFFFFu));  // no wrap-around
    // TMEM columns of a 512-column allocation; the lane field does not matter here
    EXPECT(tmem_cols(0, 32, 512) && tmem_cols(480, 32, 512) && tmem_cols((96u << 16) | 480, 32, 512));
    EXPECT(!tmem_cols(481, 32, 512) && !tmem_cols(512, 1, 512) && !tmem_cols(384, 256, 512));
    EXPECT(tmem_cols(256, 256, 512));
    // TMEM lanes: warp w reaches lanes 32 (w mod 4) .. +31
    EXPECT(tmem_lanes(0u, 4) && tmem_lanes(32u << 16, 5) && tmem_lanes(96u << 16, 11));
    EXPECT(!tmem_lanes(32u << 16, 4) && !tmem_lanes(0u, 7) && !tmem_lanes(64u << 16, 3));
    // N of a kind::f16 instruction descriptor (N / 8 in bits 17-22)
    EXPECT(idesc_n((128u >> 3) << 17) == 128 && idesc_n((64u >> 3) << 17) == 64 && idesc_n(((256u >> 3) << 17) | (8u << 24)) == 256);
    // smem descriptor start address: 16-byte units in bits 0-13
    EXPECT(desc_addr(0x1234ull | (1ull << 46)) == 0x12340u);
    // the recorded site word
    EXPECT(site(TMEM_COLS, 0x12345678u) == ((3u << 24) | 0x345678u));
    std::printf(fails ? "%d failures\n" : "ok\n", fails);
    return fails != 0;
}
"""


def test_check_predicates_on_host(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "pred.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "pred"
    subprocess.run([cxx, "-std=c++17", "-O1", f"-I{CSRC}", str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
