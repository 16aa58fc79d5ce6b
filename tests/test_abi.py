"""CPU tests of the C-ABI boundary: the library loads, exports every declared
symbol, and its host-side logic (argument checks, planner, status strings)
behaves as include/sgemm.h states.  No call here launches a kernel."""
import ctypes
import os
import re

import pytest

import sgemm_row_major_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sgemm.h")

FAKE = 1 << 20        # 16-byte aligned fake device address (never dereferenced here)
FAKE_ODD = FAKE + 4   # 4-byte aligned only


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(sgemm\w*)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from sgemm_row_major_gb300 import build
    build.build()
    return sg.load()


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("sgemm", "sgemm_status_string", "sgemm_last_cuda_error", "sgemm_sync_status", "sgemm_plan",
              "sgemm_set_variant_override", "sgemm_selftest_wait_timeout"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libsgemm.so does not export {name}"


def test_invalid_arguments_rejected_without_launch(lib):
    # (transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc) -> status
    cases = [
        (("X", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -1),
        (("N", "?", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -2),
        (("N", "N", -1, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -3),
        (("N", "N", 4, -2, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -4),
        (("N", "N", 4, 4, -3, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -5),
        (("N", "N", 4, 4, 4, 1.0, None, 4, FAKE, 4, 0.0, FAKE, 4), -7),
        (("N", "N", 4, 4, 8, 1.0, FAKE, 7, FAKE, 4, 0.0, FAKE, 4), -8),   # lda < K
        (("T", "N", 9, 4, 4, 1.0, FAKE, 8, FAKE, 4, 0.0, FAKE, 4), -8),   # lda < M for 'T'
        (("N", "N", 4, 4, 4, 1.0, FAKE, 4, None, 4, 0.0, FAKE, 4), -9),
        (("N", "N", 4, 6, 4, 1.0, FAKE, 4, FAKE, 5, 0.0, FAKE, 6), -10),  # ldb < N
        (("N", "T", 4, 4, 6, 1.0, FAKE, 6, FAKE, 5, 0.0, FAKE, 4), -10),  # ldb < K for 'T'
        (("N", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, None, 4), -12),
        (("N", "N", 4, 6, 4, 1.0, FAKE, 4, FAKE, 6, 0.0, FAKE, 5), -13),  # ldc < N
    ]
    for args, want in cases:
        assert sg.sgemm(*args, stream=0, raise_on_error=False) == want, (args, want)
        assert "invalid argument" in sg.sgemm_status_string(want)
        # the caller-workspace entry points check arguments 1-13 the same way, before any device use
        assert sg.sgemm_ex(*args, FAKE, 1 << 20, stream=0, raise_on_error=False) == want, (args, want)
        assert lib.sgemm_workspace_size(*[a.encode() if isinstance(a, str) else a for a in args],
                                        ctypes.byref(ctypes.c_size_t())) == want, (args, want)


def test_workspace_entry_points_own_arguments(lib):
    ok = ("N", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4)
    raw = [a.encode() if isinstance(a, str) else a for a in ok]
    assert lib.sgemm_workspace_size(*raw, None) == -14                      # bytes is NULL
    assert sg.sgemm_ex(*ok, FAKE_ODD, 1 << 20, stream=0, raise_on_error=False) == -14  # workspace misaligned
    for code in (-14, -15):
        assert "sgemm_ex" in sg.sgemm_status_string(code)
    # empty problems need no workspace and launch nothing
    empty = ("N", "N", 0, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4)
    assert sg.sgemm_ex(*empty, None, 0, stream=0) == 0
    assert sg.sgemm_workspace_size(*empty) == 0


def test_null_operands_allowed_when_not_read(lib):
    # M == 0 or N == 0: nothing to do, no device needed, pointers never inspected
    assert sg.sgemm("N", "N", 0, 5, 5, 1.0, None, 5, None, 5, 0.0, None, 5, stream=0) == 0
    assert sg.sgemm("N", "N", 5, 0, 5, 1.0, None, 5, None, 1, 0.0, None, 1, stream=0) == 0
    # alpha == 0: A and B are not read, so NULL is valid (planning only)
    p = sg.sgemm_plan("N", "N", 8, 8, 8, 0.0, None, 8, None, 8, 2.0, FAKE, 8, sm_count=152)
    assert p["variant_name"] == "SCALE" and p["kernel_launches"] == 1


def test_status_strings(lib):
    assert sg.sgemm_status_string(0) == "SGEMM_OK"
    for code in (1, 2, 3, 4):
        assert sg.sgemm_status_string(code).startswith("SGEMM_ERR")
    assert sg.sgemm_last_cuda_error() == 0


def plan(ta, tb, M, N, K, A=FAKE, B=FAKE, lda=None, ldb=None, sm=152, alpha=1.0):
    lda = lda if lda is not None else ((M if ta == "T" else K) or 1)
    ldb = ldb if ldb is not None else ((K if tb == "T" else N) or 1)
    return sg.sgemm_plan(ta, tb, M, N, K, alpha, A, lda, B, ldb, 0.0, FAKE, max(N, 1), sm_count=sm)


def test_planner_variants(lib):
    assert plan("N", "N", 0, 10, 10)["variant_name"] == "NONE"
    assert plan("N", "N", 10, 10, 0)["variant_name"] == "SCALE"
    big = plan("N", "N", 4096, 4096, 4096)
    assert big["variant_name"] == "TC_PRESPLIT" and big["grid_x"] == 152 and big["grid_y"] == 1
    assert (big["tile_m"], big["tile_n"], big["tile_k"], big["threads"]) == (256, 256, 32, 320)
    assert big["smem_bytes"] <= 227 * 1024
    # fewer than 4/5 as many 256 x 256 tiles as clusters (2048 x 1536: 48 < 60.8): CTA pairs with
    # 256 x 128 tiles; 2048^3 (64 tiles) splits its operands
    pair = plan("N", "N", 2048, 1536, 2048)
    assert pair["variant_name"] == "TC_PAIR" and (pair["tile_m"], pair["tile_n"], pair["threads"]) == (256, 128, 608)
    assert plan("N", "N", 2048, 2048, 2048)["variant_name"] == "TC_PRESPLIT"
    # fewer pair tiles than clusters (1024^3: 32 < 76), or M <= 128: one CTA per 128 x 128 tile
    one = plan("N", "N", 1024, 1024, 1024)
    assert one["variant_name"] == "TC_TF32X3" and one["tile_m"] == one["tile_n"] == 128
    assert plan("N", "N", 128, 65536, 1024)["variant_name"] == "TC_TF32X3"
    assert plan("N", "N", 129, 128 * 76, 64)["variant_name"] == "TC_PAIR"
    assert plan("N", "N", 129, 128 * 75, 64)["variant_name"] == "TC_TF32X3"
    # unaligned base or ld not a multiple of 4: the generic (edge) kernel up to 2 * 640^3 FLOP, the
    # split-operand kernel (whose split pass rewrites the operands aligned) from there on
    assert plan("N", "N", 512, 512, 512, A=FAKE_ODD)["variant_name"] == "GENERIC"
    assert plan("N", "N", 512, 512, 513, lda=515)["variant_name"] == "GENERIC"
    assert plan("T", "T", 512, 512, 512, ldb=514)["variant_name"] == "GENERIC"
    assert plan("N", "N", 640, 640, 639, A=FAKE_ODD)["variant_name"] == "GENERIC"
    assert plan("N", "N", 640, 640, 640, A=FAKE_ODD)["variant_name"] == "TC_PRESPLIT"
    assert plan("N", "N", 1000, 1300, 700, lda=701)["variant_name"] == "TC_PRESPLIT"
    assert plan("T", "T", 4096, 4096, 4096, ldb=4097)["variant_name"] == "TC_PRESPLIT"
    # ... unless CTA pairs cannot run (the split-operand kernel is a CTA-pair kernel)
    assert dplan("N", "N", 2048, 2048, 2048, 152, 0, A=FAKE_ODD)["variant_name"] == "GENERIC"
    # ragged padded shapes of the transpose sweep keep the TMA-fed path (ld % 4 == 0)
    for ta, tb, lda, ldb in (("N", "N", 2060, 3008), ("N", "T", 2060, 2060), ("T", "N", 4104, 3008),
                             ("T", "T", 4104, 2060)):
        assert plan(ta, tb, 4097, 3001, 2053, lda=lda, ldb=ldb)["variant_name"] == "TC_PRESPLIT"


def test_planner_split_k(lib):
    # the FFMA kernels split K into grid.y slices when the tiles cannot fill the SMs:
    # 1024^3 with 128x128 tiles -> 64 tiles, 2 slices
    try:
        sg.sgemm_set_variant_override("TMA_128x128", 0)
        p = plan("N", "N", 1024, 1024, 1024)
        assert p["split_k"] == 2 and p["kernel_launches"] == 2 and p["grid_y"] == 2
        assert p["workspace_bytes"] == 2 * 1024 * 1024 * 4
        # short-M tiles: 64x256 tiles, 16 of them -> 9 slices
        sg.sgemm_set_variant_override("TMA_64x256", 0)
        f = plan("N", "N", 64, 4096, 16384)
        assert f["variant_name"] == "TMA_64x256" and f["grid_x"] == 16 and f["split_k"] == 9
        # never more slices than K tiles, and every slice non-empty
        sg.sgemm_set_variant_override("GENERIC", 0)
        t = plan("N", "N", 8, 8, 64)
        assert t["split_k"] <= 4
        # more SMs never reduce the split
        assert plan("N", "N", 256, 256, 8192, sm=304)["split_k"] >= plan("N", "N", 256, 256, 8192)["split_k"]
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


def test_planner_stream_k(lib):
    """The one-CTA tensor-core kernel's persistent schedule: whole-tile rounds, then stream-K."""
    sg.sgemm_set_variant_override("TC_TF32X3", 0)
    try:
        _one_cta_schedules()
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


def _one_cta_schedules():
    # 4096^3: 1024 tiles on 152 SMs = 6.74 rounds -> 912 whole tiles, then the 112 tiles of the
    # ragged last round by stream-K (94 K tiles per CTA: a tile shared by up to 3 CTAs)
    p = plan("N", "N", 4096, 4096, 4096)
    assert (p["grid_x"], p["grid_y"], p["dp_tiles"], p["sk_tiles"]) == (152, 1, 912, 112)
    assert p["sk_iters"] == 112 * 128 and p["kernel_launches"] == 2 and p["split_k"] == 3
    # a remainder whose share would be short (153 tiles, 1 left over): the last round joins stream-K
    e = plan("N", "N", 128 * 17, 128 * 9, 4096)
    assert (e["dp_tiles"], e["sk_tiles"]) == (0, 153)
    assert p["workspace_bytes"] == 2 * 152 * 128 * 128 * 4
    # a whole number of rounds: whole tiles only, one launch, no workspace
    w = plan("N", "N", 128 * 19, 128 * 16, 512)
    assert (w["dp_tiles"], w["sk_tiles"], w["kernel_launches"], w["workspace_bytes"]) == (304, 0, 1, 0)
    # a ragged last round whose stream-K share would be short (K = 64): whole tiles, ragged rounds
    r = plan("N", "N", 128 * 20, 128 * 16, 64)
    assert (r["grid_x"], r["dp_tiles"], r["sk_tiles"], r["kernel_launches"]) == (152, 320, 0, 1)
    # fewer tiles than SMs with long K: stream-K over all of them on every SM
    s = plan("N", "N", 64, 4096, 16384)
    assert (s["grid_x"], s["dp_tiles"], s["sk_tiles"], s["sk_iters"]) == (152, 0, 32, 32 * 512)
    assert s["split_k"] > 1 and s["kernel_launches"] == 2
    # fewer tiles than SMs with short K: S = min(SMs / tiles, K tiles / 4) CTAs per tile
    assert plan("N", "N", 1024, 1024, 1024)["grid_x"] == 64 * 2
    t = plan("N", "N", 300, 260, 700)
    assert t["grid_x"] == 9 * 5 and t["sk_tiles"] == 9 and t["split_k"] >= 5
    q = plan("N", "N", 1000, 1300, 700)      # 88 tiles, 22 K tiles: one CTA per tile
    assert (q["grid_x"], q["split_k"], q["kernel_launches"], q["workspace_bytes"]) == (88, 1, 1, 0)
    # at least 3/4 as many tiles as SMs: whole tiles, one CTA each, no stream-K (144 of 152)
    h = plan("N", "N", 128 * 12, 128 * 12, 4096)
    assert (h["grid_x"], h["dp_tiles"], h["sk_tiles"], h["kernel_launches"]) == (144, 144, 0, 1)
    g = plan("N", "N", 128 * 12, 128 * 9, 4096)  # 108 tiles: below 3/4, stream-K
    assert (g["dp_tiles"], g["sk_tiles"], g["kernel_launches"]) == (0, 108, 2)
    # one tile, one K tile: one CTA, no fixup
    o = plan("N", "N", 128, 128, 32)
    assert (o["grid_x"], o["kernel_launches"], o["workspace_bytes"]) == (1, 1, 0)
    # a forced split: S CTAs per tile
    try:
        sg.sgemm_set_variant_override("TC_TF32X3", 5)
        f = plan("N", "N", 150, 260, 1000)
        assert f["grid_x"] == 6 * 5 and f["dp_tiles"] == 0 and f["split_k"] >= 5
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


def test_variant_override(lib):
    try:
        sg.sgemm_set_variant_override("GENERIC", 3)
        p = plan("N", "N", 4096, 4096, 4096)
        assert p["variant_name"] == "GENERIC" and p["split_k"] == 3
        sg.sgemm_set_variant_override("TMA_64x256", 0)
        assert plan("N", "N", 4096, 4096, 4096)["variant_name"] == "TMA_64x256"
        # a forced TMA variant falls back when alignment forbids it
        assert plan("N", "N", 4096, 4096, 4096, A=FAKE_ODD)["variant_name"] == "GENERIC"
        with pytest.raises(sg.SgemmError):
            sg.sgemm_set_variant_override(99, 0)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert plan("N", "N", 4096, 4096, 4096)["variant_name"] == "TC_PRESPLIT"


def test_split_operand_rule(lib):
    """TC_PRESPLIT when the split pass is amortized (>= 128 FLOP per byte it moves) and every cluster
    gets a 256 x 256 tile; CTA pairs otherwise."""
    assert plan("N", "N", 8192, 4096, 1024)["variant_name"] == "TC_PRESPLIT"
    assert plan("N", "N", 16384, 1024, 4096)["variant_name"] == "TC_PRESPLIT"
    for ta, tb in (("N", "T"), ("T", "N"), ("T", "T")):
        assert plan(ta, tb, 4096, 4096, 4096)["variant_name"] == "TC_PRESPLIT"
    # 64 products of 512x1024x1024, each operand split for two or four tiles: 60 FLOP per split byte
    assert bplan("N", "N", 512, 1024, 1024, 64, 512 * 1024, 1024 * 1024, 512 * 1024)["variant_name"] == "TC_PAIR"
    # the same products sharing one B (split once): 176 FLOP per split byte
    assert bplan("N", "N", 2048, 1024, 1024, 32, 2048 * 1024, 0, 2048 * 1024)["variant_name"] == "TC_PRESPLIT"
    # split arrays above 4 GiB (A and B 2 GiB each): CTA pairs
    assert plan("N", "N", 16384, 16384, 32768)["variant_name"] == "TC_PAIR"
    # 2048^3: 64 tiles of 256 x 256 for 76 clusters, whole tiles (no stream-K slots)
    w = plan("N", "N", 2048, 2048, 2048)
    assert (w["variant_name"], w["grid_x"], w["dp_tiles"], w["sk_tiles"]) == ("TC_PRESPLIT", 128, 64, 0)
    assert w["workspace_bytes"] == 4 * 2048 * 2048 * 4
    # workspace: stream-K slots of 128 x 256 floats per CTA, then hi and lo of A and B
    p = plan("N", "N", 8192, 4096, 1024)
    slots = 2 * 152 * 128 * 256 * 4 if p["split_k"] > 1 else 0
    assert p["workspace_bytes"] == slots + 2 * 8192 * 1024 * 4 + 2 * 4096 * 1024 * 4


def test_short_side_planner(lib):
    """TC_SKINNY for one short side (<= 64) once the long side is >= 2048 and L * K >= 2^24: tiles of
    128 along the long side, the one-CTA stream-K schedule, slots of 128 x 64 floats, the short
    operand's hi and lo arrays, and a launch for its split pass."""
    p = plan("N", "N", 64, 4096, 16384)
    assert (p["variant_name"], p["tile_m"], p["tile_n"], p["threads"]) == ("TC_SKINNY", 128, 64, 640)
    assert (p["grid_x"], p["dp_tiles"], p["sk_tiles"], p["kernel_launches"]) == (152, 0, 32, 3)
    slots = 2 * 152 * 128 * 64 * 4
    assert p["workspace_bytes"] == slots + 2 * 64 * 16384 * 4
    for ta, tb in (("N", "T"), ("T", "N"), ("T", "T")):
        assert plan(ta, tb, 64, 4096, 16384)["variant_name"] == "TC_SKINNY"
        assert plan(ta, tb, 4096, 33, 4096)["variant_name"] == "TC_SKINNY"
    assert plan("N", "N", 4096, 64, 4096)["variant_name"] == "TC_SKINNY"
    # whole tiles when they fill the SMs: 16384 x 64, K = 1024 -> 128 tiles of 128 on 152 SMs
    w = plan("N", "N", 16384, 64, 1024)
    assert (w["variant_name"], w["dp_tiles"], w["sk_tiles"], w["kernel_launches"]) == ("TC_SKINNY", 128, 0, 2)
    assert w["workspace_bytes"] == 2 * 64 * 1024 * 4
    # below the rule: a long side of 1024, a short side of 65, L * K < 2^24, a batch
    assert plan("N", "N", 1024, 64, 16384)["variant_name"] == "TC_TF32X3"
    assert plan("N", "N", 65, 4096, 16384)["variant_name"] != "TC_SKINNY"
    assert plan("N", "N", 64, 4096, 2048)["variant_name"] == "TC_TF32X3"
    assert bplan("N", "N", 64, 4096, 16384, 2, 64 * 16384, 16384 * 4096, 64 * 4096)["variant_name"] != "TC_SKINNY"
    # the long operand not TMA-aligned: not this kernel (the short one may be anything)
    assert plan("N", "N", 64, 4096, 16384, ldb=4097)["variant_name"] != "TC_SKINNY"
    assert plan("N", "N", 64, 4096, 16384, lda=16385)["variant_name"] == "TC_SKINNY"
    # no split arrays (sgemm_noalloc's planner): the one-CTA kernel
    sg.sgemm_set_variant_override("TC_SKINNY", 0)
    try:
        assert plan("N", "N", 64, 4096, 16384)["variant_name"] == "TC_SKINNY"
        assert plan("N", "N", 100, 4096, 16384)["variant_name"] == "TC_TF32X3"
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


def test_split_operand_workspace_layout(lib):
    """Workspace of TC_PRESPLIT: stream-K slots (2 per CTA, 128 x 256 floats) when a tile is shared,
    then hi and lo of op(A) and op(B) as rows of round4(K) floats, one copy per product whose operand
    differs, each part rounded up to 256 bytes."""
    def r256(x):
        return (x + 255) // 256 * 256
    sg.sgemm_set_variant_override("TC_PRESPLIT", 0)
    try:
        # K = 1001 -> rows of 1004 floats; 6 products sharing A (stride 0)
        M, N, K, batch = 300, 520, 1001, 6
        b = bplan("N", "N", M, N, K, batch, 0, 1004 * N, M * N, lda=1004, ldb=N)
        assert b["variant_name"] == "TC_PRESPLIT"
        slots = 2 * b["grid_x"] * 128 * 256 * 4 if b["kernel_launches"] == 4 else 0
        a_part, b_part = r256(1 * M * 1004 * 4), r256(batch * N * 1004 * 4)
        assert b["workspace_bytes"] == r256(slots) + 2 * a_part + 2 * b_part
        # one tile, no sharing: no slots, three launches (two split passes and the GEMM)
        one = plan("N", "N", 256, 256, 64)
        assert (one["variant_name"], one["kernel_launches"]) == ("TC_PRESPLIT", 3)
        assert one["workspace_bytes"] == 2 * r256(256 * 64 * 4) + 2 * r256(256 * 64 * 4)
        # outside the split pass's grid limits (K / 32 > 65535, more than 65535 products): CTA pairs
        assert plan("N", "N", 512, 512, 32 * 65536)["variant_name"] == "TC_PAIR"
        assert bplan("N", "N", 256, 256, 32, 65536, 256 * 32, 32 * 256, 256 * 256)["variant_name"] == "TC_PAIR"
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


def test_plan_rejects_huge_dimensions(lib):
    with pytest.raises(sg.SgemmError) as e:
        plan("N", "N", 1 << 31, 8, 8, lda=8, ldb=8)
    assert e.value.status == 4


def bplan(ta, tb, M, N, K, batch, sA, sB, sC, lda=None, ldb=None, ldc=None, A=FAKE, B=FAKE, C=FAKE, sm=152,
          alpha=1.0):
    lda = lda or (M if ta == "T" else K)
    ldb = ldb or (K if tb == "T" else N)
    ldc = ldc or N
    return sg.sgemm_plan_strided_batched(ta, tb, M, N, K, alpha, A, lda, B, ldb, 0.0, C, ldc, sA, sB, sC, batch, sm)


def test_batched_planner(lib):
    # 64 FC products of 512x1024x1024: 16 pair tiles each, one persistent launch of 76 clusters over
    # all 1024 pair tiles
    p = bplan("N", "N", 512, 1024, 1024, 64, 512 * 1024, 1024 * 1024, 512 * 1024)
    assert p["variant_name"] == "TC_PAIR" and p["grid_x"] == 152
    assert p["dp_tiles"] + p["sk_tiles"] == 64 * 16 and p["sk_tiles"] == 76 + 64 * 16 % 76
    # shared weight (stride 0) keeps the tensor-core path
    assert bplan("N", "N", 512, 1024, 1024, 8, 512 * 1024, 0, 512 * 1024)["variant_name"] == "TC_PRESPLIT"
    assert bplan("N", "N", 512, 1024, 1024, 4, 512 * 1024, 0, 512 * 1024)["variant_name"] == "TC_TF32X3"
    # few tiles in all: stream-K over the tiles of every product
    s = bplan("N", "N", 64, 4096, 16384, 2, 64 * 16384, 0, 64 * 4096)
    assert s["grid_x"] == 152 and s["sk_tiles"] == 64 and s["split_k"] > 1
    assert s["workspace_bytes"] == 2 * 152 * 128 * 128 * 4
    # one product plans exactly like sgemm()
    one = bplan("N", "N", 64, 4096, 16384, 1, 0, 0, 0)
    single = plan("N", "N", 64, 4096, 16384)
    assert one == single
    # strides that break 16-byte alignment, or overlapping operands, take the any-alignment kernel
    assert bplan("N", "N", 64, 64, 64, 4, 64 * 64 + 2, 64 * 64, 64 * 64)["variant_name"] == "GENERIC"
    assert bplan("N", "N", 64, 64, 64, 4, 64 * 32, 64 * 64, 64 * 64)["variant_name"] == "GENERIC"
    # empty batches and alpha == 0
    assert bplan("N", "N", 64, 64, 64, 0, 0, 0, 0)["variant_name"] == "NONE"
    assert bplan("N", "N", 64, 64, 64, 3, 0, 0, 64 * 64, alpha=0.0)["variant_name"] == "SCALE"


def test_small_product_planner(lib):
    """The FP32 FFMA small-product kernel is chosen by override only (batches of small products go to
    the tensor cores, two to a tile); its own rules decide where it applies."""
    def small(*a, **k):
        return bplan(*a, **k)["variant_name"] == "SMALL"
    assert bplan("N", "N", 64, 64, 64, 8192, 64 * 64, 64 * 64, 64 * 64)["variant_name"] == "TC_GROUPED"
    try:
        sg.sgemm_set_variant_override("SMALL", 0)
        # 8192 products of 64x64x64: a persistent grid of 64-thread CTAs, four per SM, no workspace
        p = bplan("N", "N", 64, 64, 64, 8192, 64 * 64, 64 * 64, 64 * 64)
        assert p["variant_name"] == "SMALL" and (p["grid_x"], p["grid_y"], p["threads"]) == (4 * 152, 1, 64)
        assert (p["kernel_launches"], p["split_k"], p["workspace_bytes"]) == (1, 1, 0)
        assert p["smem_bytes"] == 2 * 2 * 64 * 32 * 4 and p["stages"] == 2 and p["tile_k"] == 32
        # the persistent grid never exceeds the batch
        assert bplan("N", "N", 64, 64, 64, 200, 64 * 64, 64 * 64, 64 * 64)["grid_x"] == 200
        assert bplan("N", "N", 64, 64, 64, 200, 64 * 64, 64 * 64, 64 * 64, sm=1)["grid_x"] == 4
        # every op combination, ragged M and N below the tile, shared operands, any batch and K
        for ta in "NT":
            for tb in "NT":
                assert small(ta, tb, 36, 20, 100, 304, 36 * 100, 100 * 20, 36 * 20), (ta, tb)
        assert small("N", "N", 64, 64, 64, 500, 64 * 64, 0, 64 * 64)
        assert small("N", "N", 64, 64, 2048, 2, 64 * 2048, 2048 * 64, 64 * 64)
        assert plan("N", "N", 64, 64, 64)["variant_name"] == "SMALL"
        # outputs above 64, the float4 rules (contiguous extent of each operand a multiple of 4),
        # alignment of A, B, lda and strides: the any-alignment kernel
        assert bplan("N", "N", 65, 64, 64, 8192, 65 * 64, 64 * 64, 65 * 64)["variant_name"] == "GENERIC"
        assert not small("N", "N", 64, 64, 62, 8192, 64 * 64, 64 * 64, 64 * 64, lda=64)
        assert not small("N", "N", 64, 62, 64, 8192, 64 * 64, 64 * 64, 64 * 64, ldb=64)
        assert not small("T", "N", 62, 64, 64, 8192, 64 * 64, 64 * 64, 64 * 64, lda=64)
        assert not small("N", "T", 64, 64, 62, 8192, 64 * 64, 64 * 64, 64 * 64, lda=64, ldb=64)
        assert small("T", "T", 64, 62, 64, 8192, 64 * 64, 64 * 64, 64 * 64, ldb=64)
        assert bplan("N", "N", 64, 64, 64, 8192, 64 * 64, 64 * 64, 64 * 64, A=FAKE_ODD)["variant_name"] == "GENERIC"
        assert bplan("N", "N", 64, 64, 64, 8192, 64 * 66, 64 * 64, 64 * 64, lda=66)["variant_name"] == "GENERIC"
        assert bplan("N", "N", 64, 64, 64, 8192, 64 * 64 + 2, 64 * 64, 64 * 64)["variant_name"] == "GENERIC"
        # C is written with scalar stores when it is not 16-byte aligned: no rule on C
        assert small("N", "N", 64, 64, 64, 8192, 64 * 64, 64 * 64, 64 * 64 + 1, C=FAKE_ODD)
        # a CTA's (product, K chunk) items must fit an int: 2300 products x 2^25 chunks do not
        huge_k = 32 << 25
        assert bplan("N", "N", 64, 64, huge_k, 1 << 20, 0, 0, 64 * 64, lda=huge_k)["variant_name"] == "GENERIC"
        assert small("N", "N", 64, 64, huge_k, 4, 0, 0, 64 * 64, lda=huge_k)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


def test_grouped_planner(lib):
    # 2048 products of 64x64x1024: 1024 block-diagonal pairs on one persistent CTA per SM, no stream-K
    p = bplan("N", "N", 64, 64, 1024, 2048, 64 * 1024, 1024 * 64, 64 * 64)
    assert p["variant_name"] == "TC_GROUPED" and (p["grid_x"], p["threads"]) == (152, 608)
    assert (p["dp_tiles"], p["sk_tiles"], p["split_k"], p["kernel_launches"], p["workspace_bytes"]) == (1024, 0, 1, 1, 0)
    assert (p["tile_m"], p["tile_n"], p["tile_k"]) == (64, 64, 32)
    # every op combination, ragged M and N, odd batch, shared operands
    for ta in "NT":
        for tb in "NT":
            assert bplan(ta, tb, 36, 20, 300, 305, 36 * 300, 300 * 20, 36 * 20)["variant_name"] == "TC_GROUPED"
            assert bplan(ta, tb, 36, 20, 64, 305, 36 * 64, 64 * 20, 36 * 20)["variant_name"] == "TC_GROUPED"
    assert bplan("N", "T", 64, 64, 512, 400, 0, 64 * 512, 64 * 64)["variant_name"] == "TC_GROUPED"
    # fewer products than SMs, M or N above 64, TMA rules broken
    assert bplan("N", "N", 64, 64, 1024, 152, 64 * 1024, 1024 * 64, 64 * 64)["variant_name"] == "TC_GROUPED"
    assert bplan("N", "N", 64, 64, 1024, 151, 64 * 1024, 1024 * 64, 64 * 64)["variant_name"] == "TC_TF32X3"
    assert bplan("N", "N", 65, 64, 1024, 2048, 65 * 1024, 1024 * 64, 65 * 64)["variant_name"] == "TC_TF32X3"
    assert bplan("N", "N", 64, 65, 1024, 2048, 64 * 1024, 1024 * 68, 64 * 65, ldb=68)["variant_name"] == "TC_TF32X3"
    assert bplan("N", "N", 64, 64, 1024, 2048, 64 * 1024 + 2, 1024 * 64, 64 * 64)["variant_name"] == "GENERIC"
    # M, N <= 32: four products to a tile (32x32 blocks); an odd batch rounds the tiles up
    quad = bplan("N", "N", 32, 32, 32, 8193, 32 * 32, 32 * 32, 32 * 32)
    assert (quad["variant_name"], quad["tile_m"], quad["tile_n"], quad["dp_tiles"]) == ("TC_GROUPED", 32, 32, 2049)
    assert bplan("T", "T", 20, 28, 64, 1000, 20 * 64, 64 * 28, 20 * 28)["tile_m"] == 32
    assert bplan("N", "N", 33, 32, 32, 8192, 33 * 32, 32 * 32, 33 * 32)["tile_m"] == 64
    assert bplan("N", "N", 32, 33, 32, 8192, 32 * 32, 32 * 36, 32 * 33, ldb=36)["tile_m"] == 64
    # fewer SMs: fewer CTAs, the same pairs
    q = bplan("N", "N", 64, 64, 1024, 2048, 64 * 1024, 1024 * 64, 64 * 64, sm=100)
    assert (q["variant_name"], q["grid_x"], q["dp_tiles"]) == ("TC_GROUPED", 100, 1024)
    try:
        sg.sgemm_set_variant_override("TC_GROUPED", 0)
        one = plan("N", "N", 64, 64, 64)
        assert (one["variant_name"], one["grid_x"], one["dp_tiles"]) == ("TC_GROUPED", 1, 1)
        assert bplan("N", "N", 64, 64, 64, 3, 64 * 64, 64 * 64, 64 * 64)["dp_tiles"] == 2
        assert plan("N", "N", 65, 64, 64)["variant_name"] == "GENERIC"
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


def test_batched_argument_checks(lib):
    def st(sA, sB, sC, batch, M=4, N=4, ldc=4):
        return lib.sgemm_plan_strided_batched(b"N", b"N", M, N, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, ldc, sA, sB,
                                              sC, batch, 152, ctypes.byref(sg.PlanStruct()))
    assert st(16, 16, 16, 3) == 0
    assert st(-1, 16, 16, 3) == -14
    assert st(16, -1, 16, 3) == -15
    assert st(16, 16, -1, 3) == -16
    assert st(16, 16, 15, 3) == -16          # C matrices would overlap: (M-1)*ldc + N = 16
    assert st(16, 16, 0, 1) == 0             # one product: strideC is never used
    assert st(16, 16, 16, -1) == -17
    assert lib.sgemm_plan_strided_batched(b"N", b"N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4, 16, 16, 16, 3,
                                          152, None) == -19
    # the sgemm() checks come first, with the same argument numbers
    assert lib.sgemm_plan_strided_batched(b"N", b"N", 4, 4, 8, 1.0, FAKE, 7, FAKE, 4, 0.0, FAKE, 4, 16, 16, 16, 3,
                                          152, ctypes.byref(sg.PlanStruct())) == -8
    # and the entry point itself rejects before touching a device
    assert lib.sgemm_strided_batched(b"N", b"N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4, 16, 16, 15, 3,
                                     None) == -16
    assert sg.sgemm_status_string(-17).startswith("invalid argument 17")


def dplan(ta, tb, M, N, K, sm_count, pair_clusters, A=FAKE, B=FAKE):
    lda = M if ta == "T" else K
    ldb = K if tb == "T" else N
    return sg.sgemm_plan_for_device(ta, tb, M, N, K, 1.0, A, lda, B, ldb, 0.0, FAKE, N, sm_count, pair_clusters)


def test_planner_for_device_pair_clusters(lib):
    """The co-resident CTA-pair cluster count steers the planner: SMs / 2 gives sgemm_plan()'s plan;
    fewer clusters (an SM limit) size the pair grid; none leaves the CTA-pair kernels out, and a
    forced one falls back to one CTA per tile."""
    for shape in ((4096, 4096, 4096), (2048, 2048, 2048), (1000, 1300, 700), (8192, 4096, 1024)):
        assert dplan("N", "N", *shape, 152, 76) == plan("N", "N", *shape)
    p = dplan("N", "N", 4096, 4096, 4096, 152, 60)
    assert p["variant_name"] == "TC_PRESPLIT" and p["grid_x"] == 120
    for shape in ((4096, 4096, 4096), (2048, 2048, 2048), (8192, 4096, 1024)):
        p = dplan("N", "N", *shape, 152, 0)
        assert p["variant_name"] == "TC_TF32X3" and p["grid_x"] <= 152, shape
    try:
        for v in ("TC_PAIR", "TC_PRESPLIT"):
            sg.sgemm_set_variant_override(v, 0)
            assert dplan("N", "N", 4096, 4096, 4096, 152, 0)["variant_name"] == "TC_TF32X3"
            assert dplan("N", "N", 4096, 4096, 4096, 152, 0, A=FAKE_ODD)["variant_name"] == "GENERIC"
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    # argument checks of the device description
    for bad_sm, bad_pc, code in ((0, 76, -14), (152, -1, -15)):
        with pytest.raises(sg.SgemmError) as ei:
            dplan("N", "N", 64, 64, 64, bad_sm, bad_pc)
        assert ei.value.status == code
    st = lib.sgemm_plan_for_device(b"N", b"N", 64, 64, 64, 1.0, FAKE, 64, FAKE, 64, 0.0, FAKE, 64, 152, 76, None)
    assert st == -16


def test_tf32_planner(lib):
    """sgemm_tf32: rounded copies of op(A) and op(B) (one part each, rows of round4(K) floats)
    after the stream-K slots, two rounding passes, the CTA-pair GEMM, the fixup when tiles are
    shared; any alignment; no CTA-pair device: unsupported."""
    def r256(x):
        return (x + 255) // 256 * 256
    p = sg.sgemm_tf32_plan("N", "N", 4096, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, 0.0, FAKE, 4096, 152)
    assert (p["variant_name"], p["tile_m"], p["tile_n"], p["grid_x"], p["stages"]) == ("TC_TF32", 256, 256, 152, 6)
    slots = 2 * 152 * 128 * 256 * 4 if p["split_k"] > 1 else 0
    assert p["workspace_bytes"] == r256(slots) + 2 * 4096 * 4096 * 4
    assert p["kernel_launches"] == (4 if p["split_k"] > 1 else 3)
    q = sg.sgemm_tf32_plan("T", "N", 333, 277, 501, 1.0, FAKE_ODD, 335, FAKE_ODD, 279, 0.0, FAKE, 277, 152)
    assert q["variant_name"] == "TC_TF32"
    assert q["workspace_bytes"] % 256 == 0 and q["workspace_bytes"] >= r256(333 * 504 * 4) + r256(277 * 504 * 4)
    assert sg.sgemm_tf32_plan("N", "N", 64, 64, 0, 1.0, FAKE, 1, FAKE, 64, 0.0, FAKE, 64, 152)["variant_name"] == "SCALE"
    with pytest.raises(sg.SgemmError) as ei:
        sg.sgemm_tf32_plan("N", "N", 64, 64, 32 * 65536, 1.0, FAKE, 32 * 65536, FAKE, 64, 0.0, FAKE, 64, 152)
    assert ei.value.status == sg.STATUS["ERR_UNSUPPORTED"]


def test_bf16_planner(lib):
    """sgemm_bf16: BF16 copies of op(A) and op(B) (rows of round8(K) two-byte values) after the
    stream-K slots, two rounding passes, the CTA-pair GEMM on 64-deep K tiles, the fixup when tiles
    are shared; any alignment; the same shape limits as sgemm_tf32."""
    def r256(x):
        return (x + 255) // 256 * 256
    p = sg.sgemm_bf16_plan("N", "N", 4096, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, 0.0, FAKE, 4096, 152)
    assert (p["variant_name"], p["tile_m"], p["tile_n"], p["tile_k"], p["grid_x"], p["stages"]) == \
        ("TC_BF16", 256, 256, 64, 152, 6)
    slots = 2 * 152 * 128 * 256 * 4 if p["split_k"] > 1 else 0
    assert p["workspace_bytes"] == r256(slots) + 2 * 4096 * 4096 * 2
    assert p["kernel_launches"] == (4 if p["split_k"] > 1 else 3)
    # stream-K for the ragged last round only (28 of 256 tiles: 16 of the 64-deep K tiles per
    # cluster is enough), never the last whole round with it (K = 1024: whole tiles)
    assert (p["dp_tiles"], p["sk_tiles"]) == (228, 28) and p["split_k"] > 1
    fc = sg.sgemm_bf16_plan("N", "N", 8192, 4096, 1024, 1.0, FAKE, 1024, FAKE, 4096, 0.0, FAKE, 4096, 152)
    assert (fc["dp_tiles"], fc["sk_tiles"], fc["split_k"]) == (512, 0, 1)
    q = sg.sgemm_bf16_plan("T", "N", 333, 277, 501, 1.0, FAKE_ODD, 335, FAKE_ODD, 279, 0.0, FAKE, 277, 152)
    assert q["variant_name"] == "TC_BF16"
    assert q["workspace_bytes"] % 256 == 0 and q["workspace_bytes"] >= r256(333 * 504 * 2) + r256(277 * 504 * 2)
    assert sg.sgemm_bf16_plan("N", "N", 64, 64, 0, 1.0, FAKE, 1, FAKE, 64, 0.0, FAKE, 64, 152)["variant_name"] == "SCALE"
    assert sg.sgemm_bf16_plan("N", "N", 0, 64, 64, 1.0, FAKE, 64, FAKE, 64, 0.0, FAKE, 64, 152)["variant_name"] == "NONE"
    with pytest.raises(sg.SgemmError) as ei:
        sg.sgemm_bf16_plan("N", "N", 64, 64, 32 * 65536, 1.0, FAKE, 32 * 65536, FAKE, 64, 0.0, FAKE, 64, 152)
    assert ei.value.status == sg.STATUS["ERR_UNSUPPORTED"]


def test_debug_library_exports_every_declared_symbol():
    """libsgemm_debug.so (the bounds-checking build) exports the same entry points and reports
    itself; libsgemm.so has the checks compiled out."""
    from sgemm_row_major_gb300 import build
    build.build(debug=True)
    dbg = sg.load_debug()
    for name in declared_functions():
        assert hasattr(dbg, name), f"libsgemm_debug.so does not export {name}"
    assert dbg.sgemm_debug_bounds_enabled() == 1
    assert sg.load().sgemm_debug_bounds_enabled() == 0
    assert "SGEMM_ERR_BOUNDS" in sg.sgemm_status_string(sg.STATUS["ERR_BOUNDS"])
