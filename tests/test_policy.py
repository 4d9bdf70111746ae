"""The library's automatic host-side choices, checked on the CPU: the FFMA
kernel's K-split of the tiles after its last full round (the per-SM model),
the transpose rule for K-major fp32 operands, the row panels that
gemm_host() pipelines its copies over, and the tensor-core kernel's tile
shape and last-round split. tests/policy_probe.cc is compiled with
the host C++ compiler against the library's own policy header, so these are
the choices the library makes; the expected values are the outcomes the
model gives by hand for a 152-SM GB300 (two FFMA CTAs per SM), including the
shapes whose splits were measured (2560x2048x8192: 8 slices;
4096x2048x2048: 2; 1024x1024x8192: 7; 8192^3 and 2048^3: none)."""

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "dense_gemm_06_gb300", "csrc")
P, SLOTS = 152, 304  # SMs, resident FFMA CTAs (two per SM)


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("policy") / "policy_probe")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "policy_probe.cc"),
                    "-o", exe], check=True, capture_output=True, text=True)

    def run(*args):
        out = subprocess.run([exe, *map(str, args)], check=True, capture_output=True, text=True)
        vals = [int(v) for v in out.stdout.split()]
        return vals[0] if len(vals) == 1 else tuple(vals)
    return run


def tiles(M, N):
    return ((M + 127) // 128) * ((N + 127) // 128)


@pytest.mark.parametrize("M,N,K,want", [
    # 320 tiles: 2 full rounds + 16; s in 2..8 adds 1/s of a round -> 8 slices
    (2560, 2048, 8192, (304, 8, 64)),
    # 512 tiles: 3 rounds + 56; 128 k-tiles allow s <= 4; s = 2 saves 12.5%
    (4096, 2048, 2048, (456, 2, 64)),
    # 64 tiles, no full round: 7 slices take 3/7 of a round
    (1024, 1024, 8192, (0, 7, 74)),
    # 4096 tiles: 26 rounds + 144 -- no split saves a round
    (8192, 8192, 8192, (4096, 1, 512)),
    # exactly one full round: the model does not hold there, never split
    (2048, 2048, 2048, (256, 1, 128)),
    # a whole number of rounds: nothing to split
    (2432, 2048, 4096, (304, 1, 256)),
    # 9 rounds + 100: even the best split saves less than 10%
    (1468 * 128, 128, 8192, (1468, 1, 512)),
    # 64 tiles but only 40 k-tiles: no slice would keep 32 k-tiles
    (1024, 1024, 640, (64, 1, 40)),
])
def test_tail_split_automatic(probe, M, N, K, want):
    assert probe("split", tiles(M, N), SLOTS, P, (K + 15) // 16, 0) == want


def test_tail_split_never_and_forced(probe):
    assert probe("split", 320, SLOTS, P, 512, 1) == (320, 1, 512)
    # forced (tests): the last wave of resident CTAs in 2..4 slices
    assert probe("split", 320, SLOTS, P, 512, 2) == (304, 4, 128)   # 16 tail tiles
    assert probe("split", 64, SLOTS, P, 512, 2) == (0, 4, 128)      # under one wave
    assert probe("split", 608, SLOTS, P, 512, 2) == (304, 2, 256)   # whole waves
    assert probe("split", 1000, SLOTS, P, 7, 2) == (912, 3, 3)      # 88 tail tiles
    # occupancy unknown: never
    assert probe("split", 320, 0, P, 512, 0) == (320, 1, 512)
    assert probe("split", 0, SLOTS, P, 512, 0) == (0, 1, 512)


def test_transpose_rule(probe):
    assert probe("transpose", 8192, 8192, 8192, 8192, 0) == 1
    assert probe("transpose", 511, 8192, 511, 8192, 0) == 0      # other dimension < 512
    assert probe("transpose", 1024, 1024, 1024, 2047, 0) == 0    # M N K just below 2^31
    assert probe("transpose", 1024, 1024, 1024, 2048, 0) == 1    # M N K = 2^31
    assert probe("transpose", 8192, 8192, 8192, 8192, 1) == 0    # never
    assert probe("transpose", 4, 4, 4, 4, 2) == 1                # always


def test_host_panels(probe):
    # fp32 8192^3: 304 CTA slots, 64 tile columns -> 19 tile rows per panel
    # (a whole number of waves), so 8192 rows go as 2432 x 3 + 896
    assert probe("panel", 8192, 8192, 8192, 1, 2, 2, 1, P) == 2432
    # bf16 8192^3 on 76 CTA pairs (256 x 256 tiles): 19 tile rows of 256
    assert probe("panel", 8192, 8192, 8192, 0, 2, 2, 1, P) == 4864
    # one CTA per 128 x 256 tile: 152 slots, 32 tile columns -> 19 rows of 128
    assert probe("panel", 8192, 8192, 8192, 0, 2, 1, 1, P) == 2432
    # clusters of two pairs (512-row tiles): 19 tile rows exceed the 16 there
    assert probe("panel", 8192, 8192, 8192, 0, 2, 2, 2, P) == 8192
    # the FFMA slots per SM matter: 18 tile columns, 304 vs 152 slots
    assert probe("panel", 16384, 2304, 8192, 1, 2, 2, 1, P) == 16384
    assert probe("panel", 16384, 2304, 8192, 1, 1, 2, 1, P) == 9728
    # more than 8 panels' worth of waves: the wave count is doubled
    assert probe("panel", 400000, 128, 1000, 1, 2, 2, 1, P) == 77824
    # too small to pipeline (M N K < 1e10), or nothing to multiply
    assert probe("panel", 2048, 2048, 2048, 1, 2, 2, 1, P) == 2048
    assert probe("panel", 8192, 8192, 0, 1, 2, 2, 1, P) == 8192


@pytest.mark.parametrize("M,N,cg,tn,mc,want", [
    # 1024 x 512: 8 pair tiles < 152 / 4 -> one CTA per tile, 8 x 8 tiles of 64
    (1024, 512, 0, 0, 0, (1, 64)),
    # 16 x 16 pair tiles >= 38: CTA pairs, 256 wide
    (4096, 4096, 0, 0, 0, (2, 256)),
    # the ragged fp16 problem (16 x 12 pair tiles) and the skinny one (64)
    (4095, 3071, 0, 0, 0, (2, 256)),
    (16384, 256, 0, 0, 0, (2, 256)),
    # 37 pair tiles (37 x 4 < 152): one CTA per tile; 74 row tiles x 4 of 64
    # columns would not fit one round over 152 SMs, x 2 of 128 do (148)
    (256 * 37, 256, 0, 0, 0, (1, 128)),
    # 74 pair tiles (296 >= 152): CTA pairs
    (128 * 74, 512, 0, 0, 0, (2, 256)),
    # forced values win; a pair needs 128 columns at least; multicast is 2 x 256
    (1024, 512, 2, 0, 0, (2, 256)),
    (1024, 512, 2, 64, 0, (2, 128)),
    (8192, 8192, 1, 0, 0, (1, 256)),
    (8192, 8192, 0, 128, 0, (2, 128)),
    (1024, 512, 1, 0, 1, (2, 256)),
])
def test_tc_shape(probe, M, N, cg, tn, mc, want):
    assert probe("tcshape", M, N, cg, tn, mc, P) == want


def test_tc_split(probe):
    # bf16 8192^3: 1024 pair tiles on 76 pairs, last round 36 <= 38 -> split
    assert probe("tcsplit", 1024, 76, 256, 2, 0, 0) == 988
    # ragged fp16: 192 tiles, last round 40 > 38 -> no gain, no split
    assert probe("tcsplit", 192, 76, 256, 2, 0, 0) == 192
    # one round or less, a whole number of rounds: no split
    assert probe("tcsplit", 64, 76, 256, 2, 0, 0) == 64
    assert probe("tcsplit", 152, 76, 256, 2, 0, 0) == 152
    # half units must keep 64 columns per CTA; multicast never splits
    assert probe("tcsplit", 1024, 76, 128, 2, 0, 0) == 1024
    assert probe("tcsplit", 1024, 76, 256, 2, 1, 0) == 1024
    assert probe("tcsplit", 400, 152, 128, 1, 0, 0) == 400   # 96 in the last round > 76
    assert probe("tcsplit", 350, 152, 128, 1, 0, 0) == 304   # 46 in the last round
    # never / forced (tests: the last round, or every tile under one round)
    assert probe("tcsplit", 1024, 76, 256, 2, 0, 1) == 1024
    assert probe("tcsplit", 192, 76, 256, 2, 0, 2) == 152
    assert probe("tcsplit", 8, 76, 256, 2, 0, 2) == 0
    assert probe("tcsplit", 152, 76, 256, 2, 0, 2) == 76
    # occupancy unknown: never
    assert probe("tcsplit", 1024, 0, 256, 2, 0, 0) == 1024


def test_stream_k(probe):
    # fp32 2048^3: 256 tiles on 152 SMs (304 slots): every tile's iterations
    # shared by 304 stream-K CTAs (two tiles' time -> 1.68)
    assert probe("sk", 256, SLOTS, P, 128, 0) == (0, 304)
    # 1.8 P (273.6) is the break-even of the 10% rule; 2 P or more: none
    assert probe("sk", 273, SLOTS, P, 128, 0) == (0, 304)
    assert probe("sk", 274, SLOTS, P, 128, 0) == (274, 0)
    assert probe("sk", 304, SLOTS, P, 128, 0) == (304, 0)
    # under one tile per SM (the K-slice rule's case), too few k-tiles, one
    # CTA per SM only, or another mode: none
    assert probe("sk", 151, SLOTS, P, 128, 0) == (151, 0)
    assert probe("sk", 256, SLOTS, P, 31, 0) == (256, 0)
    assert probe("sk", 256, P, P, 128, 0) == (256, 0)
    assert probe("sk", 256, SLOTS, P, 128, 1) == (256, 0)
    assert probe("sk", 256, SLOTS, P, 128, 2) == (256, 0)
    # forced (tests): a third whole, the rest over 3/2 as many CTAs as tiles,
    # never more CTAs than iterations
    assert probe("sk", 30, SLOTS, P, 64, 3) == (10, 30)
    assert probe("sk", 7, SLOTS, P, 64, 3) == (2, 8)
    assert probe("sk", 4, SLOTS, P, 1, 3) == (1, 3)


def test_host_k_pieces(probe):
    # fp32 C with several panels: the first panel in 4 pieces of whole 64-deep
    # k-tiles (the last piece takes the remainder)
    assert probe("kpieces", 4, 4, 8192) == (4, 0, 2048, 4096, 6144, 8192)
    assert probe("kpieces", 2, 4, 1037) == (4, 0, 320, 576, 832, 1037)
    assert probe("kpieces", 2, 4, 1024) == (4, 0, 256, 512, 768, 1024)
    # one panel, a 16-bit C (rounded between pieces), or K under 4 x 256: whole
    assert probe("kpieces", 1, 4, 8192) == (1, 0, 8192)
    assert probe("kpieces", 4, 2, 8192) == (1, 0, 8192)
    assert probe("kpieces", 4, 4, 1023) == (1, 0, 1023)
    # every K from 1024 up: bounds increase, every piece but the last is a
    # whole number of 64-deep k-tiles, and the pieces cover [0, K)
    for K in list(range(1024, 1300)) + [4095, 8191, 65537]:
        n, *b = probe("kpieces", 3, 4, K)
        assert n == 4 and b[0] == 0 and b[-1] == K
        assert all(b[j] < b[j + 1] for j in range(n)), (K, b)
        assert all(b[j] % 64 == 0 for j in range(n)), (K, b)
