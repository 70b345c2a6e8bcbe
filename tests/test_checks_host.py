"""The predicates of the checked build (csrc/checks.h), compiled with g++ on
the host and called through ctypes: each rule accepts the accesses the
kernels make and rejects the ones it exists to catch."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "exact_tiled_attention_10_gb300", "csrc", "checks.h")

SHIM = r'''
#include "checks.h"
extern "C" {
int tma_inner_ok(long long x, int e) { return fa::chk::tma_inner_ok(x, e); }
int tma_store_ok(long long x, long long y, int e) { return fa::chk::tma_store_ok(x, y, e); }
int sw128_base_ok(unsigned a) { return fa::chk::sw128_base_ok(a); }
int bulk_ok(unsigned long long d, unsigned long long s, unsigned n) { return fa::chk::bulk_ok(d, s, n); }
int tmem_ok(unsigned t, unsigned n, unsigned w) { return fa::chk::tmem_ok(t, n, w); }
int range_ok(long long o, long long n, long long s) { return fa::chk::range_ok(o, n, s); }
int tile_ok(long long h, long long hs, long long t, long long ts) { return fa::chk::tile_ok(h, hs, t, ts); }
unsigned check_mask() { return fa::kErrCheckMask; }
unsigned check_bits() { return fa::kErrCheckTma | fa::kErrCheckTmem | fa::kErrCheckSmem | fa::kErrCheckTile; }
}
// the predicates are usable in constant expressions (compile-time checks)
static_assert(fa::chk::tma_inner_ok(64, 1) && !fa::chk::tma_inner_ok(8, 1), "");
static_assert(fa::chk::tmem_ok(0, 512, 0) && !fa::chk::tmem_ok(1, 512, 0), "");
'''


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("no g++")
    d = tmp_path_factory.mktemp("checks")
    src, so = d / "shim.cpp", d / "libshim.so"
    src.write_text(SHIM)
    subprocess.run(["g++", "-std=c++17", "-O1", "-shared", "-fPIC", "-I", os.path.dirname(HDR), str(src), "-o",
                    str(so)], check=True)
    return ctypes.CDLL(str(so))


def test_tma_inner_coordinate(lib):
    # multiples of 16 bytes pass: 16 elements of any size, 8 bf16, 4 float32
    assert lib.tma_inner_ok(0, 1) and lib.tma_inner_ok(64, 1) and lib.tma_inner_ok(96, 4)
    assert lib.tma_inner_ok(8, 2) and lib.tma_inner_ok(4, 4) and lib.tma_inner_ok(-64, 2)
    # the faulting ones: an odd half-tile, 4 bf16 (8 bytes), 8 one-byte codes
    assert not lib.tma_inner_ok(4, 2) and not lib.tma_inner_ok(8, 1) and not lib.tma_inner_ok(33, 4)
    # what the kernels issue: boxes at 0 / 64 of the head dim, dQ quarters at 32 q, K^T at key blocks
    for x in (0, 32, 64, 96, 128 * 7):
        assert lib.tma_inner_ok(x, 1)


def test_tma_store_coordinates(lib):
    assert lib.tma_store_ok(32, 4096, 4)
    assert not lib.tma_store_ok(-32, 0, 4)  # a store never starts left of the tensor
    assert not lib.tma_store_ok(0, -1, 4)
    assert not lib.tma_store_ok(2, 0, 4)


def test_swizzle_base_and_bulk(lib):
    assert lib.sw128_base_ok(0) and lib.sw128_base_ok(1024 * 37)
    assert not lib.sw128_base_ok(512) and not lib.sw128_base_ok(1024 + 16)
    assert lib.bulk_ok(0x1000, 0x7f0000000010, 512)
    assert not lib.bulk_ok(0x1008, 0x10, 512) and not lib.bulk_ok(0x10, 0x14, 512)
    assert not lib.bulk_ok(0x10, 0x10, 500) and not lib.bulk_ok(0x10, 0x10, 0)


def test_tmem_quadrant_and_columns(lib):
    lane = lambda l: l << 16
    # warp w reaches lanes 32 (w % 4) .. +31; 512 columns in all
    assert lib.tmem_ok(lane(0) | 0, 128, 0) and lib.tmem_ok(lane(64) | 384, 128, 6)
    assert lib.tmem_ok(lane(96) | 480, 32, 11)
    assert not lib.tmem_ok(lane(32) | 0, 32, 0)   # another warp's quadrant
    assert not lib.tmem_ok(lane(0) | 496, 32, 4)  # runs past column 511
    assert not lib.tmem_ok(lane(128) | 0, 16, 4)  # no lane 128


def test_ranges_and_tiles(lib):
    assert lib.range_ok(0, 16, 16) and lib.range_ok(8176, 16, 8192)
    assert not lib.range_ok(8180, 16, 8192) and not lib.range_ok(-4, 4, 64) and not lib.range_ok(0, -1, 64)
    assert lib.tile_ok(0, 1, 0, 1) and lib.tile_ok(31, 32, 15, 16)
    assert not lib.tile_ok(32, 32, 0, 16) and not lib.tile_ok(0, 32, 16, 16) and not lib.tile_ok(-1, 32, 0, 1)


def test_check_bits_do_not_overlap_the_wait_bits(lib):
    bits = lib.check_bits()
    assert bits == lib.check_mask()
    assert bits & 0xFFFF == 0  # the wait time-out bits live below bit 16
