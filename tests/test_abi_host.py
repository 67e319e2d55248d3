"""The C-ABI library on the host (no GPU needed): it loads, exports what the
header declares, plans exactly by the pages' closed forms, and rejects bad
arguments before making any CUDA call."""
from __future__ import annotations

import ctypes
import math

import pytest

import dense_tensor_core_bf16_gb300 as g
from dense_tensor_core_bf16_gb300 import _build
from oracle import plan_forms as pf


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build_library()
    g.lib()


GB300 = dict(num_sms=152, smem_per_sm=233472, smem_optin_per_cta=232448, smem_reserved_per_cta=1024,
             regs_per_sm=65536, max_threads_per_sm=2048, max_ctas_per_sm=32, tmem_cols_per_sm=512)


def dev(**over):
    d = dict(GB300)
    d.update(over)
    return g.gemm_device_desc_t(**d)


def test_exports_every_declared_function():
    names = g.header_functions()
    assert len(names) >= 12
    L = g.lib()
    for n in names:
        assert hasattr(L, n), n
    for n in names:
        assert n in g.__all__, f"binding lacks {n}"


def test_binding_structs_match_the_header(tmp_path):
    """Every struct the binding mirrors has the size and field offsets the C
    compiler gives it from include/gemm_bf16.h."""
    import subprocess
    structs = {"gemm_device_desc_t": g.gemm_device_desc_t, "gemm_kernel_desc_t": g.gemm_kernel_desc_t,
               "gemm_plan_t": g.gemm_plan_t, "gemm_options_t": g.gemm_options_t,
               "gemm_epilogue_t": g.gemm_epilogue_t, "gemm_conv2d_desc_t": g.gemm_conv2d_desc_t,
               "gemm_host_problem_t": g.gemm_host_problem_t}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "gemm_bf16.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{name}.{field} %zu\\n", offsetof({name}, {field}));')
    lines.append("  return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", _build.INCLUDE, "-o", str(exe), str(src)])
    out = dict(l.rsplit(" ", 1) for l in subprocess.check_output([str(exe)], text=True).splitlines())
    for name, cls in structs.items():
        assert int(out[name]) == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert int(out[f"{name}.{field}"]) == getattr(cls, field).offset, f"{name}.{field}"


def test_status_and_limiter_strings():
    assert g.gemm_status_string(0) == "GEMM_OK"
    assert g.gemm_status_string(7) == "GEMM_ERR_DEVICE_TIMEOUT"
    assert [g.gemm_limiter_string(i) for i in range(5)] == ["registers", "smem", "tmem", "threads", "blocks"]


def test_occupancy_worked_example_through_the_abi():
    """230,400 B and 155 registers x 256 threads: one CTA per SM, registers
    binding first, and still one with no shared memory at all."""
    d = dev(smem_per_sm=227 * 1024, smem_reserved_per_cta=0, tmem_cols_per_sm=512)
    k = g.gemm_kernel_desc_t(regs_per_thread=155, threads_per_cta=256, smem_per_cta=230400, tmem_cols_per_cta=0)
    assert g.gemm_occupancy(k, d) == (0, 1, "registers")
    k0 = g.gemm_kernel_desc_t(regs_per_thread=155, threads_per_cta=256, smem_per_cta=0, tmem_cols_per_cta=0)
    assert g.gemm_occupancy(k0, d) == (0, 1, "registers")
    # 128 registers x 256 threads = 32,768: two fit by registers; smem still allows one
    k2 = g.gemm_kernel_desc_t(regs_per_thread=128, threads_per_cta=256, smem_per_cta=230400, tmem_cols_per_cta=0)
    assert g.gemm_occupancy(k2, d) == (0, 1, "smem")
    k3 = g.gemm_kernel_desc_t(regs_per_thread=32, threads_per_cta=256, smem_per_cta=1000, tmem_cols_per_cta=256)
    assert g.gemm_occupancy(k3, d) == (0, 2, "tmem")
    bad = g.gemm_kernel_desc_t(regs_per_thread=32, threads_per_cta=0, smem_per_cta=0, tmem_cols_per_cta=0)
    assert g.gemm_occupancy(bad, d)[0] == 1


def kern(variant, regs=64, max_active_clusters=0):
    """The library's own footprint of a variant, with a register count."""
    k = g.gemm_kernel_desc(variant)
    k.regs_per_thread = regs
    k.max_active_clusters = max_active_clusters
    return k


def _plan(M, N, K, split=1, persistent=1, d=None, regs=64, out=g.GEMM_OUT_BF16, variant=1, mac=0, no_sk=0):
    o = g.options(split_k=split, non_persistent=0 if persistent else 1, kernel_variant=variant, no_stream_k=no_sk)
    st, p = g.gemm_plan_for_device(M, N, K, g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, out, o, d or dev(),
                                   kern(variant, regs, mac))
    assert st == 0
    return p


WORKLOADS = [(256, 256, 256), (4096, 4096, 4096), (4095, 4096, 4096), (4097, 4096, 4096),
             (4096, 4096, 4088), (4096, 4104, 4096), (3968, 4096, 4096), (16384, 8192, 8192),
             (128, 256, 65536), (1, 1, 1), (129, 257, 65)]
TILES = {1: (128, 256, 1), 2: (256, 256, 2), 3: (256, 128, 2), 4: (128, 128, 1)}
TILE_K = {1: 64, 2: 128, 3: 64, 4: 64}


def test_kernel_desc_without_a_device():
    for v, (tm, tn, cs) in TILES.items():
        k = g.gemm_kernel_desc(v)
        assert k.threads_per_cta == 192 and k.cluster_size == cs
        assert 0 < k.smem_per_cta <= 232448
        assert k.tmem_cols_per_cta == 2 * tn      # two accumulators of tn fp32 columns (a power of two)


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
@pytest.mark.parametrize("S,mac", [(148, 0), (152, 0), (152, 72)])
@pytest.mark.parametrize("shape", WORKLOADS)
def test_plan_matches_oracle_closed_forms(shape, S, mac, variant):
    """The plan against the oracle's closed forms; S b is the number of CTAs
    resident at once (for two-CTA tiles: resident clusters times two)."""
    M, N, K = shape
    tm, tn, cs = TILES[variant]
    k = kern(variant, 64, mac)
    p = _plan(M, N, K, d=dev(num_sms=S), variant=variant, mac=mac)
    b, lim = pf.ctas_per_sm(regs_per_thread=64, threads=192, smem_per_cta=k.smem_per_cta, regs_per_sm=65536,
                            smem_per_sm=233472, smem_reserved_per_cta=1024)
    assert (p.ctas_per_sm, g.LIMITERS[p.occupancy_limiter]) == (b, lim) == (1, "smem")
    clusters = S * b // cs
    if mac:
        clusters = min(clusters, mac)
    R = clusters * cs
    assert p.resident_ctas == R and p.cluster_size == cs and p.kernel_variant == variant
    tk = TILE_K[variant]
    assert (p.tile_m, p.tile_n, p.tile_k) == (tm, tn, tk)
    assert p.tiles == pf.grid(M, N, tm, tn)
    assert p.grid == pf.grid(M, N, tm, tn, p.split_k) * cs
    assert p.eta_wave == pytest.approx(float(pf.eta_wave(p.grid, R, 1)), rel=1e-15)
    assert p.eta_pad == pytest.approx(float(pf.eta_pad(M, N, K, tm, tn, tk)), rel=1e-15)
    assert p.flops == pf.flops(M, N, K)
    assert (p.m_padded, p.n_padded, p.k_padded) == (pf.padded(M, tm), pf.padded(N, tn), pf.padded(K, tk))
    assert p.launch_ctas == min(p.grid, R)
    assert p.k_tiles == math.ceil(K / tk)


def test_plan_hand_values_148_sms():
    d = dev(num_sms=148)
    p = _plan(4096, 4096, 4096, d=d)
    assert (p.grid, p.launch_ctas) == (512, 148)
    assert p.eta_wave == pytest.approx(512 / 592, rel=1e-15)
    p = _plan(4097, 4096, 4096, d=d)
    assert p.eta_pad == pytest.approx(4097 / 4224, rel=1e-15)
    p = _plan(4096, 4096, 4096, persistent=0, d=d)
    assert p.launch_ctas == 512 and p.persistent == 0


def test_plan_hand_values_pair_tiles_152_sms():
    """256x256 pair tiles: 16 x 16 = 256 tiles, 512 CTAs on 152 resident CTAs
    = 4 rounds (608 slots).  256x128: 512 tiles, 1024 CTAs, 7 rounds (1064)."""
    p = _plan(4096, 4096, 4096, variant=2)
    assert (p.tiles, p.grid, p.resident_ctas, p.launch_ctas) == (256, 512, 152, 152)
    assert p.eta_wave == pytest.approx(512 / 608, rel=1e-15)
    p = _plan(4096, 4096, 4096, variant=3)
    assert (p.tiles, p.grid) == (512, 1024)
    assert p.eta_wave == pytest.approx(1024 / 1064, rel=1e-15)
    # 72 resident pairs (some SMs without a partner): 144 CTAs, 4 rounds of 144
    p = _plan(4096, 4096, 4096, variant=2, mac=72)
    assert p.resident_ctas == 144 and p.eta_wave == pytest.approx(512 / 576, rel=1e-15)
    p = _plan(16384, 8192, 8192, variant=2)
    assert (p.tiles, p.grid) == (2048, 4096)
    assert p.eta_wave == pytest.approx(4096 / (27 * 152), rel=1e-15)


@pytest.mark.parametrize("split,eta", [(1, 1 / 148), (8, 8 / 148), (32, 32 / 148), (74, 0.5), (148, 1.0)])
def test_plan_split_k_workload(split, eta):
    p = _plan(128, 256, 65536, split=split, d=dev(num_sms=148), out=g.GEMM_OUT_F32)
    assert p.split_k == split and p.grid == split
    assert p.eta_wave == pytest.approx(eta, rel=1e-15)
    assert p.eta_pad == 1.0
    assert p.k_tiles == 1024 and p.k_tiles_per_split == math.ceil(1024 / split)
    assert p.workspace_bytes == (split * 128 * 256 * 4 if split > 1 else 0)


def test_plan_at_the_size_limits():
    """K = 2^31 - 8 for one output, and a C of more than 2^31 elements: the
    plans the GPU size-limit tests run, by hand.  One tile of 2^25 64-wide
    k-tiles splits over the 152 single CTAs (each slice at least 4 k-tiles);
    the pair kernel with a forced tail spreads its one tile over all 76
    clusters; the large C has 513 x 129 single-CTA tiles of one k-tile."""
    K = (1 << 31) - 8
    p = _plan(1, 1, K, split=0, out=g.GEMM_OUT_F32)
    assert p.k_tiles == (K + 63) // 64 == 1 << 25
    assert p.split_k == 152 and p.k_tiles_per_split == -(-(1 << 25) // 152)
    assert p.workspace_bytes == 152 * 128 * 256 * 4
    p = _plan(1, 1, K, split=0, variant=2, mac=76, no_sk=-1, out=g.GEMM_OUT_F32)
    assert p.k_tiles == 1 << 24 and p.stream_k_tiles == 1 and p.dp_tiles == 0 and p.split_k == 1
    assert p.launch_ctas == 152 and p.workspace_bytes == 76 * 256 * 256 * 4
    p = _plan(1, 1, K, split=1, variant=2, mac=76, out=g.GEMM_OUT_F32)
    assert p.split_k == 1 and p.stream_k_tiles == 0 and p.launch_ctas == 2
    M, N = 65605, 32792
    assert M * N > 1 << 31
    p = _plan(M, N, 72, split=0)
    assert (p.tiles, p.k_tiles, p.split_k, p.stream_k_tiles) == (513 * 129, 2, 1, 0)


def test_plan_split_k_clamped_and_auto():
    p = _plan(128, 256, 200, split=50)        # 4 k-tiles: at most 4 slices
    assert p.split_k == 4
    p = _plan(128, 256, 65536, split=0)       # auto: one tile, 1024 k-tiles, 152 slots
    assert p.split_k == 152
    p = _plan(128, 256, 65536, split=0, variant=2)   # pairs: 76 slots
    assert p.split_k == 76 and p.grid == 152
    p = _plan(4096, 4096, 4096, split=0)      # auto: the tiles fill the GPU, no split
    assert p.split_k == 1


def test_plan_auto_variant():
    """Equal balanced work (4096^3: 216 k-tiles per cluster either way) goes to
    the pair kernel; M = 128 with a long K goes to the 128 x 128 single-CTA
    kernel: two tiles, the plan's own split 152 / 2 = 76, 152 CTAs in one wave."""
    st, p = g.gemm_plan_for_device(4096, 4096, 4096, 0, 1, 1, None, dev(), kern(2))
    assert st == 0 and p.kernel_variant == 2
    st, _ = g.gemm_plan_for_device(4096, 4096, 4096, 0, 1, 1, None, dev(), kern(1))
    assert st == 1     # a footprint that does not match the variant
    st, p = g.gemm_plan_for_device(128, 256, 65536, 0, 1, 0, None, dev(), kern(4))
    assert st == 0 and p.kernel_variant == 4 and p.split_k == 76
    for shape in [(16384, 8192, 8192), (4097, 4096, 4096), (3968, 4096, 4096), (2048, 2048, 1024),
                  (1536, 1536, 1536), (512, 512, 4096)]:
        st, p = g.gemm_plan_for_device(*shape, 0, 1, 1, None, dev(), kern(2))
        assert st == 0 and p.kernel_variant == 2, shape
    # small GEMMs (256 x 128 pair tiles filling at most half the pairs, K < 2048)
    # go to the 256 x 128 pair kernel
    for shape in [(256, 256, 256), (512, 512, 512), (1024, 1024, 1024), (1024, 1024, 2047)]:
        st, p = g.gemm_plan_for_device(*shape, 0, 1, 1, None, dev(), kern(3))
        assert st == 0 and p.kernel_variant == 3, shape


@pytest.mark.parametrize("shape,split,want_variant,want_split", [
    ((128, 256, 65536), 0, 4, 76),     # the plan's own split for two 128 x 128 tiles: 152 units
    ((128, 256, 65536), 74, 4, 74),    # 2 x 74 = 148 units: one wave
    ((128, 256, 65536), 32, 4, 32),
    ((128, 256, 65536), 8, 4, 8),
    ((128, 256, 65536), 1, 4, 1),      # two CTAs instead of one
    ((128, 256, 65536), 148, 1, 148),  # 2 x 148 > 152: the 128 x 256 kernel, one wave of 148
    ((128, 1024, 4096), 0, 4, 16),     # both plans split by 16: 128 units against 64
    ((100, 300, 8192), 0, 4, 32),      # ragged: three 128 x 128 tiles, 128 k-tiles at 4 per slice
    ((100, 3000, 2048), 0, 4, 1),      # 24 unsplit 128 x 128 tiles beat 12 tiles split by 8
    ((128, 4096, 2048), 0, 4, 1),      # 32 unsplit tiles: 15.3 against 19.4 us split by 8
    ((96, 512, 16384), 0, 4, 38),      # 11.4 against 12.8 us
    ((64, 1536, 4096), 0, 4, 12),
    ((128, 2048, 8192), 0, 4, 9),
    ((64, 4096, 4096), 0, 1, 9),       # only the 128 x 256 plan splits (16 tiles x 9)
    ((128, 8192, 8192), 0, 1, 4),      # likewise: 32 tiles x 4
    ((129, 256, 65536), 0, 2, 76),     # two tile rows: the rule does not apply (the pair kernel)
    ((128, 128, 65536), 0, 1, 152),    # N <= 128: one tile either way
    ((128, 256, 1024), 1, 3, 1),       # short K: the small-GEMM pair kernel
])
def test_plan_one_tile_row_with_a_long_k(shape, split, want_variant, want_split):
    """The automatic variant for a single row of tiles (M <= 128, N > 128,
    K >= 2048): the 128 x 128 single-CTA kernel when all its units fit in one
    wave and its estimated time (operand bytes per CTA at the per-SM feed,
    unique bytes at HBM rate, the split-K round trip) beats the 128 x 256
    plan's, with more units winning a near tie.  The expected choices are the
    faster plans measured on GB300 (S = 152)."""
    M, N, K = shape
    o = g.options(split_k=split)
    st, p = g.gemm_plan_for_device(M, N, K, 0, 1, 0, o, dev(), kern(want_variant))
    assert st == 0 and p.kernel_variant == want_variant and p.split_k == want_split, (p.kernel_variant, p.split_k)


def _want_stream_k(T, C, K, KB, force=False, variant=2):
    """The decomposition rule of gemm_plan_for_device for the plan's own split
    on a persistent grid: a tail of C + (T mod C) tiles (all T below 2C) when
    T mod C != 0 and it pays -- T >= C and the last wave's idle share,
    (ceil(T/C) C - T) / C k-tiles scaled to 128-wide k-tiles of a 128 x 256
    block per SM, at least 12 -- or always when forced."""
    if KB < 2 or T % C == 0:
        return 0
    tm, tn, cs = TILES[variant]
    idle = (math.ceil(T / C) * C - T) / C * KB
    waste = idle * (TILE_K[variant] / 128) * (tm * tn / cs / (128 * 256))
    if force or (T >= C and waste >= 12.0):
        return C + T % C if T >= 2 * C else T
    return 0


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("shape", WORKLOADS + [(4096, 4096, 8192), (2560, 4096, 4096), (1000, 9000, 3000),
                                                (2560, 2560, 8192), (3072, 3072, 3072), (1792, 1792, 1792)])
def test_plan_stream_k_tail(shape, variant):
    """T tiles on C clusters; the largest per-cluster share of a stream-K plan
    is ceil(dp/C) whole tiles plus ceil(sk k-iterations / C)."""
    M, N, K = shape
    tm, tn, cs = TILES[variant]
    C = 152 // cs
    T = pf.grid(M, N, tm, tn)
    KB = math.ceil(K / TILE_K[variant])
    for force in (False, True):
        p = _plan(M, N, K, split=0, variant=variant, no_sk=-1 if force else 0)
        want_sk = _want_stream_k(T, C, K, KB, force, variant)
        assert p.stream_k_tiles == want_sk and p.dp_tiles == T - want_sk, (force, T, C)
        if want_sk:
            assert p.split_k == 1 and p.launch_ctas == C * cs
            worst = math.ceil((T - want_sk) / C) * KB + math.ceil(want_sk * KB / C)
            assert p.eta_stream_k == pytest.approx(T * KB / C / worst, rel=1e-12)
            assert p.workspace_bytes == C * tm * tn * 4
        else:
            assert p.eta_stream_k == 0
    # off on request, and never on a one-CTA-per-tile grid or with an explicit split
    assert _plan(M, N, K, split=0, variant=variant, no_sk=1).stream_k_tiles == 0
    assert _plan(M, N, K, split=0, variant=variant, persistent=0, no_sk=-1).stream_k_tiles == 0
    assert _plan(M, N, K, split=1, variant=variant, no_sk=-1).stream_k_tiles == 0


@pytest.mark.parametrize("shape,variant,want", [
    ((1536, 1536, 1536), 2, 1),      # 36 pair tiles, short K: one tile per cluster
    ((1024, 1024, 4096), 2, 1),      # 16 tiles, K below 6144: no split
    ((1024, 1024, 8192), 2, 4),      # 16 tiles (16 * 4 <= 76), long K: 76 / 16 = 4 slices
    ((512, 512, 2048), 2, 4),        # 4 tiles (4 * 8 <= 76), K >= 2048: 16 k-tiles, 4 per slice
    ((512, 512, 1024), 2, 1),        # K below 2048
    ((2048, 1024, 4096), 2, 1),      # 32 tiles: 32 * 4 > 76
    ((128, 256, 65536), 1, 152),     # the split-K workload: one tile, 152 slices
])
def test_plan_automatic_split_rule(shape, variant, want):
    M, N, K = shape
    p = _plan(M, N, K, split=0, variant=variant)
    assert p.split_k == want and p.stream_k_tiles == 0


def test_plan_raster_group():
    """Raster groups of 8 m-tiles when the tiles make at least eight waves of
    the resident clusters on a persistent grid, else 16; an option wins."""
    assert _plan(16384, 8192, 8192, split=0, variant=2, mac=76).raster_group_m == 8    # 2048 tiles >= 8 x 76
    assert _plan(8192, 4864, 4096, split=0, variant=2, mac=76).raster_group_m == 8     # 32 x 19 = 608 tiles
    assert _plan(8192, 4608, 4096, split=0, variant=2, mac=76).raster_group_m == 16    # 32 x 18 = 576 tiles
    assert _plan(4096, 4096, 4096, split=0, variant=2, mac=76).raster_group_m == 16
    assert _plan(16384, 8192, 8192, split=0, variant=2, mac=76, persistent=0).raster_group_m == 16
    o = g.options(split_k=0, kernel_variant=2, raster_group_m=5)
    st, p = g.gemm_plan_for_device(16384, 8192, 8192, 0, 1, 1, o, dev(), kern(2, 64, 76))
    assert st == 0 and p.raster_group_m == 5


def test_plan_stream_k_hand_values():
    """4096^3 on 76 pairs of 256x256 tiles with 128-wide k-tiles: T = 256,
    256 mod 76 = 28, a tail of 104 tiles (3328 k-iterations, 43.8 per
    cluster) after 152 whole tiles; the largest share is 2 x 32 + 44 = 108
    k-iterations of an ideal 256 x 32 / 76 = 107.79."""
    p = _plan(4096, 4096, 4096, split=0, variant=2)
    assert (p.tiles, p.stream_k_tiles, p.dp_tiles, p.k_tiles) == (256, 104, 152, 32)
    assert p.eta_stream_k == pytest.approx((256 * 32 / 76) / 108, rel=1e-12)
    p = _plan(4096, 4096, 4096, split=0, variant=1)   # 64-wide k-tiles: 2 x ... on 152 CTAs
    assert (p.tiles, p.stream_k_tiles, p.k_tiles) == (512, 208, 64)
    assert p.eta_stream_k == pytest.approx((512 * 64 / 152) / (2 * 64 + math.ceil(208 * 64 / 152)), rel=1e-12)


def test_plan_stream_k_ranges_for_long_epilogues():
    """With a GELU epilogue or one that reads C, the stream-K tail is dealt in
    whole half tiles when k_tiles is even and at least 8.  4096^3: 104 tail
    tiles are 208 halves of 16 iterations on 76 clusters, three to the first
    56 and two to the rest (48 or 32 iterations), so the largest share is
    2 x 32 + 48 = 112 k-iterations.  4097 x 4096 x 4096: 272 tiles, a tail of
    76 + 44 = 120 tiles, 240 halves, four to the first 12 clusters: 2 x 32 +
    64 = 128.  ReLU or no activation without C keep the even ranges (108 and
    2 x 32 + 51 = 115)."""
    cases = [((4096, 4096, 4096), ("gelu", 0.0), 112), ((4096, 4096, 4096), ("gelu", 1.0), 112),
             ((4096, 4096, 4096), ("none", 1.0), 112), ((4096, 4096, 4096), ("relu", 0.0), 108),
             ((4096, 4096, 4096), ("none", 0.0), 108), ((4097, 4096, 4096), ("gelu", 1.0), 128),
             ((4097, 4096, 4096), ("relu", 0.0), 115)]
    for (M, N, K), (act, beta), worst in cases:
        epi = g.gemm_epilogue_t(alpha=1.0, beta=beta, bias=None, activation=g.ACTIVATIONS[act])
        o = g.options(split_k=0, kernel_variant=2, epilogue=ctypes.pointer(epi))
        st, p = g.gemm_plan_for_device(M, N, K, g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, g.GEMM_OUT_BF16, o,
                                       dev(), kern(2, 64, 0))
        assert st == 0 and p.k_tiles == 32 and p.stream_k_tiles == (104 if M == 4096 else 120)
        assert p.eta_stream_k == pytest.approx(p.tiles * 32 / 76 / worst, rel=1e-12), (M, act, beta)


def test_plan_takes_no_stream_k_tail_beyond_160_clusters():
    """The tail's range boundaries travel in the kernel's parameters, one per
    cluster, for at most 160 clusters: a device with more resident clusters
    (a made-up 400-SM part, one CTA per cluster) gets whole tiles or split-K,
    never a tail, even when a tail is forced."""
    big = dev(num_sms=400)
    for no_sk in (0, -1):
        p = _plan(8192, 8192, 4096, split=0, d=big, variant=1, no_sk=no_sk)
        assert p.stream_k_tiles == 0 and p.eta_stream_k == 0
    p = _plan(8192, 8192, 4096, split=0, variant=1, no_sk=-1)   # 152 clusters: the tail is there
    assert p.stream_k_tiles > 0


def test_plan_stream_k_short_k_moves_boundaries_to_tile_edges():
    """k_tiles below 8 (here 4, a reach of one iteration): a long epilogue's
    boundaries within k_tiles / 4 of a tile's edge move to the edge.  The
    3328 x 3072 x 512 tail of 80 tiles (320 iterations, 4.2 per cluster) after
    one whole tile of 4 iterations per cluster: the longest range grows from 5
    to 6, the largest share from 9 to 10; other epilogues keep 9."""
    for act, beta, worst in (("gelu", 0.0, 10), ("none", 1.0, 10), ("none", 0.0, 9), ("relu", 0.0, 9)):
        epi = g.gemm_epilogue_t(alpha=1.0, beta=beta, bias=None, activation=g.ACTIVATIONS[act])
        o = g.options(split_k=0, kernel_variant=2, no_stream_k=-1, epilogue=ctypes.pointer(epi))
        st, p = g.gemm_plan_for_device(3328, 3072, 512, g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, g.GEMM_OUT_BF16, o,
                                       dev(), kern(2, 64, 0))
        assert st == 0 and (p.tiles, p.stream_k_tiles, p.k_tiles) == (156, 80, 4)
        assert p.eta_stream_k == pytest.approx(156 * 4 / 76 / worst, rel=1e-12), (act, beta)


def _call(M, N, K, A=16, lda=64, B=16, ldb=64, C=16, ldc=64, la=0, lb=1, out=0, split=1):
    return g.gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, la, lb, out, split, None)


def test_argument_checks_before_any_cuda_call():
    # (pointers here are fake; every case must be rejected, or be a no-op, before use)
    assert _call(-1, 4, 4) == 1
    assert _call(4, 4, 1 << 31) == 1
    assert _call(4, 4, 4, la=2) == 1
    assert _call(4, 4, 4, out=5) == 1
    assert _call(4, 4, 4, split=-1) == 1
    assert _call(64, 4, 4, la=1, lda=32) == 1    # column-major A: lda < M
    assert _call(4, 64, 4, lb=0, ldb=32) == 1    # row-major B: ldb < N
    assert _call(60, 4, 4, la=1, lda=60) == 2    # column-major A: 120-byte lines
    assert _call(4, 60, 4, lb=0, ldb=60) == 2    # row-major B: 120-byte lines
    assert _call(0, 4, 4) == 0            # empty: nothing to do
    assert _call(4, 0, 4) == 0
    assert _call(4, 4, 4, C=0) == 1       # NULL C
    assert _call(4, 64, 4, ldc=32) == 1   # ldc < N
    assert _call(4, 4, 64, lda=32) == 1   # lda < K
    assert _call(4, 4, 64, A=0) == 1      # NULL A
    assert _call(4, 4, 4, A=18) == 2      # A not on 16 bytes
    assert _call(4, 4, 4, B=24) == 2
    assert _call(4, 4, 4, C=20) == 2
    assert _call(4, 4, 60, lda=60) == 2   # 120 bytes: not a multiple of 16
    assert _call(4, 4, 4, ldc=66) == 2    # fp32: 264 bytes
    assert _call(4, 4, 4, ldc=68, out=1) == 2   # bf16: 136 bytes
    opts = g.gemm_options_t(timeout_ms=-1)
    assert g.gemm_bf16_ex(4, 4, 4, 16, 64, 16, 64, 16, 64, 0, 1, 0, opts, None) == 1
    opts = g.gemm_options_t(kernel_variant=9)
    assert g.gemm_bf16_ex(4, 4, 4, 16, 64, 16, 64, 16, 64, 0, 1, 0, opts, None) == 1
    # fused epilogue: an unknown activation, a bias off its 16-byte boundary
    bad = g.gemm_epilogue_t(alpha=1.0, beta=0.0, bias=None, activation=3)
    assert g.gemm_bf16_ex(4, 4, 4, 16, 64, 16, 64, 16, 64, 0, 1, 0,
                          g.gemm_options_t(epilogue=ctypes.pointer(bad)), None) == 1
    off = g.gemm_epilogue_t(alpha=1.0, beta=1.0, bias=20, activation=1)
    assert g.gemm_bf16_ex(4, 4, 4, 16, 64, 16, 64, 16, 64, 0, 1, 0,
                          g.gemm_options_t(epilogue=ctypes.pointer(off)), None) == 2


def test_plan_argument_checks():
    k = kern(1)
    plan = g.gemm_plan_t()
    L = g.lib()
    assert L.gemm_plan_for_device(4, 4, 4, 0, 1, 0, None, None, ctypes.byref(k), ctypes.byref(plan)) == 1
    o1 = g.options(kernel_variant=1)
    # every layout pair plans the same launch
    st, p_default = g.gemm_plan_for_device(300, 500, 700, 0, 1, 0, o1, dev(), k)
    assert st == 0
    for la, lb in [(1, 1), (0, 0), (1, 0)]:
        st, p = g.gemm_plan_for_device(300, 500, 700, la, lb, 0, o1, dev(), k)
        assert st == 0 and p.as_dict() == p_default.as_dict()
    st, _ = g.gemm_plan_for_device(4, 4, 4, 0, 1, 0, g.options(kernel_variant=7), dev(), k)
    assert st == 1
    too_big = kern(1)
    too_big.smem_per_cta = 240000
    st, _ = g.gemm_plan_for_device(4, 4, 4, 0, 1, 0, o1, dev(), too_big)
    assert st == 1


def _conv(**kw):
    d = dict(N=2, H=9, W=11, C=64, K=128, R=3, S=3, pad_h=1, pad_w=1, stride_h=1, stride_w=1, dil_h=1, dil_w=1)
    d.update(kw)
    return g.gemm_conv2d_desc_t(**d)


def test_conv2d_out_dims_match_the_oracle_formula():
    import oracle
    for H in (1, 5, 9, 17):
        for R in (1, 2, 3, 5):
            for pad in (0, 1, 2):
                for stride in (1, 2, 3):
                    for dil in (1, 2):
                        st, P, Q = g.gemm_conv2d_out_dims(_conv(H=H, W=H + 3, R=R, S=R, pad_h=pad, pad_w=pad,
                                                                stride_h=stride, stride_w=stride, dil_h=dil, dil_w=dil))
                        p = oracle.conv2d_out_size(H, R, pad, stride, dil)
                        q = oracle.conv2d_out_size(H + 3, R, pad, stride, dil)
                        if p >= 1 and q >= 1:
                            assert (st, P, Q) == (0, p, q)
                        else:
                            assert st == 1


def test_conv2d_argument_checks_before_any_cuda_call():
    x, w, y = 256, 512, 768   # fake, 16-byte aligned: every case below is rejected before use
    call = lambda d, out=0, opts=None, xp=x: g.gemm_conv2d_fprop_bf16(d, xp, w, y, out, opts, None)
    assert call(_conv(N=0)) == 1
    assert call(_conv(stride_h=0)) == 1
    assert call(_conv(pad_w=-1)) == 1
    assert call(_conv(H=2, R=5, pad_h=0)) == 1                 # filter larger than the padded image
    assert call(_conv(C=60)) == 2                               # 120-byte pixel rows
    assert call(_conv(K=66)) == 2                               # fp32 output rows of 264 bytes
    assert call(_conv(K=60), out=1) == 2                        # bf16 output rows of 120 bytes
    assert call(_conv(), xp=x + 8) == 2                         # x off its 16-byte boundary
    assert call(_conv(), opts=g.options(kernel_variant=9)) == 1
    assert call(_conv(pad_h=128, H=300)) == 3                   # beyond an im2col pixel box's range
    assert call(_conv(R=65, dil_h=2, H=200)) == 3
    assert call(_conv(), opts=g.options(debug_skip_load=1)) == 1


def _host(M=4, N=4, K=8, A=16, lda=8, la=0, B=16, ldb=8, lb=1, C=16, ldc=4):
    return g.gemm_host_problem_t(M=M, N=N, K=K, A=A, lda=lda, layout_a=la, B=B, ldb=ldb, layout_b=lb, C=C, ldc=ldc)


def test_host_batch_argument_checks_before_any_cuda_call():
    """gemm_bf16_host_batch checks every problem before it enqueues anything;
    no host-side rule on alignment (the device copies are pitched)."""
    L = g.lib()
    assert L.gemm_bf16_host_batch(-1, None, 0, None, None) == 1
    assert L.gemm_bf16_host_batch(2, None, 0, None, None) == 1
    assert g.gemm_bf16_host_batch([], 0, None, None) == 0
    assert g.gemm_bf16_host_batch([_host()], 7, None, None) == 1                 # bad output type
    assert g.gemm_bf16_host_batch([_host(la=2)], 0, None, None) == 1
    assert g.gemm_bf16_host_batch([_host(M=-1)], 0, None, None) == 1
    assert g.gemm_bf16_host_batch([_host(lda=7)], 0, None, None) == 1            # row-major A: lda < K
    assert g.gemm_bf16_host_batch([_host(la=1, lda=3)], 0, None, None) == 1      # column-major A: lda < M
    assert g.gemm_bf16_host_batch([_host(lb=0, ldb=3)], 0, None, None) == 1      # row-major B: ldb < N
    assert g.gemm_bf16_host_batch([_host(ldc=3)], 0, None, None) == 1
    assert g.gemm_bf16_host_batch([_host(C=0)], 0, None, None) == 1
    assert g.gemm_bf16_host_batch([_host(A=0)], 0, None, None) == 1
    assert g.gemm_bf16_host_batch([_host(K=0, A=0, B=0)], 0, g.options(timeout_ms=-1), None) == 1
    bad = g.gemm_epilogue_t(alpha=1.0, beta=0.0, bias=None, activation=3)
    assert g.gemm_bf16_host_batch([_host()], 0, g.gemm_options_t(epilogue=ctypes.pointer(bad)), None) == 1
    # a bad problem anywhere in the batch rejects the whole batch
    assert g.gemm_bf16_host_batch([_host(M=0), _host(), _host(ldb=2)], 0, None, None) == 1
    # only empty problems: nothing to do, no device needed
    assert g.gemm_bf16_host_batch([_host(M=0), _host(N=0, C=0)], 0, None, None) == 0
