"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, rejects invalid arguments before touching CUDA, and plans work."""
import ctypes
import os
import re

import numpy as np
import pytest

from dense_bf16_gemm_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_bf16.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^GEMM_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_list():
    assert declared_symbols() == sorted(_native.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # and nothing else is exported with C linkage besides the header's symbols
    out = os.popen(f"nm -D --defined-only {_native.library_path()}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    gemm_like = {s for s in exported if s.startswith("gemm_")}
    assert gemm_like == set(declared_symbols())


def declared_prototypes():
    """name -> (return type, [parameter types]) of every GEMM_API function."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for ret, name, params in re.findall(r"GEMM_API\s+([\w\s\*]*?)\b(\w+)\s*\(([^)]*)\)\s*;",
                                        text):
        params = " ".join(params.split())
        types = [] if params in ("", "void") else [
            re.sub(r"\s*\b\w+$", "", p.strip()).replace(" *", "*") for p in params.split(",")]
        protos[name] = (" ".join(ret.split()), types)
    return protos


def _ctype_of(decl):
    """The ctypes type the binding must use for a C parameter or return type."""
    decl = decl.replace("const ", "").strip()
    if decl.endswith("*"):
        return "ptr"
    return {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "float": ctypes.c_float,
            "uint32_t": ctypes.c_uint32, "uint64_t": ctypes.c_uint64}[decl]


def test_binding_signatures_match_the_header(lib):
    """Every ctypes binding passes as many arguments as the header's prototype
    takes, each of the C type's width and kind, and reads the declared return
    type: a dropped or swapped argument in the binding fails here, not on a GPU."""
    protos = declared_prototypes()
    assert sorted(protos) == declared_symbols()
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == len(params), (name, params)
        for i, (ct, decl) in enumerate(zip(fn.argtypes, params)):
            want = _ctype_of(decl)
            if want == "ptr":
                assert ct in (ctypes.c_void_p, ctypes.c_char_p) or \
                    issubclass(ct, ctypes._Pointer), (name, i, decl, ct)
            else:
                assert ct is want, (name, i, decl, ct)
        want = _ctype_of(ret)
        if want == "ptr":
            assert fn.restype in (ctypes.c_void_p, ctypes.c_char_p), (name, ret)
        else:
            assert fn.restype is want, (name, ret, fn.restype)


def test_status_strings(lib):
    for st in range(6):
        assert _native.status_string(st)
    assert _native.status_string(99) == "unknown status"


A16 = 1 << 20   # a 16-byte aligned fake address: validation never dereferences it


@pytest.mark.parametrize("args,expect", [
    # (M, N, K, A, lda, B, ldb, C, ldc, dtype)
    ((-1, 8, 8, A16, 8, A16, 8, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),
    ((8, -1, 8, A16, 8, A16, 8, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, -1, A16, 8, A16, 8, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),
    ((1 << 31, 8, 8, A16, 8, A16, 8, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, 8, A16, 8, A16, 8, A16, 8, 7), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, 16, A16, 8, A16, 16, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),   # lda < K
    ((8, 8, 16, A16, 16, A16, 8, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),   # ldb < K
    ((8, 16, 8, A16, 8, A16, 8, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),    # ldc < N
    ((8, 8, 8, 0, 8, A16, 8, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),       # NULL A
    ((8, 8, 8, A16, 8, 0, 8, A16, 8, 1), _native.GEMM_ERR_INVALID_ARG),       # NULL B
    ((8, 8, 8, A16, 8, A16, 8, 0, 8, 1), _native.GEMM_ERR_INVALID_ARG),       # NULL C
    ((8, 8, 8, A16 + 2, 8, A16, 8, A16, 8, 1), _native.GEMM_ERR_ALIGNMENT),
    ((8, 8, 8, A16, 8, A16 + 8, 8, A16, 8, 1), _native.GEMM_ERR_ALIGNMENT),
    ((8, 8, 8, A16, 8, A16, 8, A16 + 4, 8, 1), _native.GEMM_ERR_ALIGNMENT),
    ((8, 8, 12, A16, 12, A16, 16, A16, 8, 1), _native.GEMM_ERR_ALIGNMENT),    # lda*2 % 16
    ((8, 8, 12, A16, 16, A16, 12, A16, 8, 1), _native.GEMM_ERR_ALIGNMENT),    # ldb*2 % 16
    ((8, 6, 8, A16, 8, A16, 8, A16, 6, 0), _native.GEMM_ERR_ALIGNMENT),       # ldc*4 % 16
    ((8, 12, 8, A16, 8, A16, 8, A16, 12, 1), _native.GEMM_ERR_ALIGNMENT),     # ldc*2 % 16
    ((0, 8, 8, 0, 8, 0, 8, 0, 8, 1), _native.GEMM_OK),                        # empty: no-op
    ((8, 0, 8, 0, 8, 0, 8, 0, 0, 0), _native.GEMM_OK),
])
def test_gemm_validation_without_gpu(lib, args, expect):
    M, N, K, A, lda, B, ldb, C, ldc, dt = args
    st = _native.gemm_bf16(M, N, K, 1.0, A, lda, B, ldb, 0.0, C, ldc, dt, 0)
    assert st == expect


@pytest.mark.parametrize("args,expect", [
    ((-1, 8, 8, A16, 8, A16, A16, 8, A16, 8), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, 16, A16, 8, A16, A16, 16, A16, 8), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, 8, A16, 8, 0, A16, 8, A16, 8), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, 8, A16, 8, A16, 0, 8, A16, 8), _native.GEMM_ERR_INVALID_ARG),
    ((8, 16, 8, A16, 8, A16, A16, 8, A16, 8), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, 8, A16, 8, A16, A16 + 2, 8, A16, 8), _native.GEMM_ERR_ALIGNMENT),
    ((8, 12, 8, A16, 8, A16, A16, 8, A16, 12), _native.GEMM_ERR_ALIGNMENT),
    ((8, 0, 8, 0, 8, 0, 0, 8, 0, 0), _native.GEMM_OK),
])
def test_gate_up_validation_without_gpu(lib, args, expect):
    M, N, K, X, ldx, Wg, Wu, ldw, Y, ldy = args
    assert _native.gemm_gate_up_silu(M, N, K, X, ldx, Wg, Wu, ldw, Y, ldy, 0) == expect


def test_problems_beyond_32_bit_work_units_are_refused(lib):
    """At most 2^25 blocks of 128 x 128 outputs per call (the kernels count work
    units in 32 bits, at most 32 per block); the limit sits far above what any
    GPU memory holds, so it refuses only problems that cannot exist, in the
    plans and the calls."""
    big = (1 << 31) - 1
    for batch, M, N in [(1, big, big), (1 << 20, 1 << 20, 1 << 12), ((1 << 25) + 1, 1, 1),
                        (3, 1 << 19, (1 << 20) + 1)]:
        st, _ = _native.gemm_batched_plan(batch, M, N, 64, 0, 1, 152)
        assert st == _native.GEMM_ERR_INVALID_ARG, (batch, M, N)
    st = _native.gemm_bf16(big, big, 64, 1.0, A16, 64, A16, 64, 0.0, A16, big, 1, 0)
    assert st == _native.GEMM_ERR_INVALID_ARG
    st = _native.gemm_gate_up_silu(big, big, 64, A16, 64, A16, A16, 64, A16, big, 0)
    assert st == _native.GEMM_ERR_INVALID_ARG
    # exactly 2^25 blocks is allowed, with every unit count within 32 bits
    for batch, M, N, K in [(1 << 25, 1, 1, 8192), (1, 1 << 19, 1 << 19, 64),
                           (1, big, 1 << 7, 4096), (1 << 20, 16, 1 << 12, 1 << 20)]:
        st, p = _native.gemm_batched_plan(batch, M, N, K, 0, 1, 152)
        d = p.as_dict()
        assert st == 0 and 1 <= d["grid"] <= 152, (batch, M, N, K)
        assert 1 <= d["tiles"] < (1 << 31) and 1 <= d["split_k"] <= 32, (batch, M, N, K, d)


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _native.gemm_bf16(8, 8, 8, 1.0, A16, 8, A16, 8, 0.0, A16, 8, 1, 0)
    assert st in (_native.GEMM_ERR_CUDA, _native.GEMM_ERR_UNSUPPORTED)


def balanced_division(tiles, kb, slots):
    """The balanced division restated: cluster c takes positions
    [c*per + min(c, extra), ...) of the tile-major k-block sequence.  Returns
    (units, most pieces of one tile, k-blocks of the longest range)."""
    work = tiles * kb
    per, extra = divmod(work, slots)
    starts = [c * per + min(c, extra) for c in range(slots + 1)]
    units, owners = 0, {}
    for c in range(slots):
        r0, r1 = starts[c], starts[c + 1]
        if r1 <= r0:
            continue
        for t in range(r0 // kb, (r1 - 1) // kb + 1):
            units += 1
            owners.setdefault(t, set()).add(c)
    assert sorted(owners) == list(range(tiles))       # every tile is covered
    return units, max(len(v) for v in owners.values()), -(-work // slots)


def pair_model(M, N, K, slots=76, widths=(256, 224), balanced=False, strips=True):
    """Restatement of the planner's rule: fewest waves (a split tail wave counts
    1/split + 0.1; a tail wave of 256-wide tiles that is not split along K and
    whose tiles, cut into four 64-column strips, fit on the pairs counts 0.63
    when that is fewer; with the balanced division enabled, that division where
    it applies, counting its longest range in tiles + 0.1 when a tile is cut)
    weighted by width + 320.  Returns (width, most pieces of a tile, units,
    balanced)."""
    best = None
    kb = -(-K // 64)
    for bn in widths:
        tiles = -(-M // 256) * -(-N // bn)
        full, tail = tiles - tiles % slots, tiles % slots
        split = 1
        if tail:
            s_ = min(2, slots // tail, kb // 24)
            if s_ >= 2:
                kbp = -(-kb // s_)
                split = -(-kb // kbp)
        if split == 1:
            full = tiles
        waves = full // slots + ((1 / split + 0.1) if split > 1 else (1 if tiles - full // slots * slots else 0))
        cand = (bn, split, full + (tiles - full) * split, False)
        if strips and bn == 256 and tail and split == 1 and 4 * tail <= slots:
            if tiles // slots + 0.63 < waves:
                waves = tiles // slots + 0.63
                cand = (bn, 1, tiles - tail + 4 * tail, False)
        if balanced and tiles >= slots:
            units, pieces, longest = balanced_division(tiles, kb, slots)
            waves = longest / kb + (0.1 if pieces > 1 else 0.0)
            cand = (bn, pieces, units, True)
        cost = waves * (bn + 320)
        if best is None or cost < best[0]:
            best = (cost,) + cand
    return best[1:]


def test_balanced_division_restatement():
    # 3000 x 5000 x 2000 on 256-wide tiles: 240 tiles of 32 k-blocks over 76
    # pairs, ranges of 101 or 102 k-blocks; a cut tile has two pieces
    units, pieces, longest = balanced_division(240, 32, 76)
    assert longest == 102 and pieces == 2 and 240 < units <= 240 + 75
    # whole waves: ranges end on tile boundaries, nothing is cut
    assert balanced_division(152, 10, 76) == (152, 1, 20)
    # ranges shorter than a tile: a tile falls in several ranges
    assert balanced_division(3, 100, 76)[1] >= 25


def test_plan_pair_4096(lib):
    st, p = _native.gemm_bf16_plan(4096, 4096, 4096, _native.GEMM_OUT_BF16, 152)
    assert st == 0
    d = p.as_dict()
    assert d["kernel_name"] == "pair"
    assert d["tile_m"] == 256 and d["tile_k"] == 64 and d["stages"] == 6
    # 16 x 16 = 256 pair tiles on 76 pairs: 3 whole waves, and the 28 tiles of
    # the last wave each cut into 2 K pieces (56 units) so that wave is half long
    assert d["tile_n"] == 256 and d["split_k"] == 2
    assert d["tiles"] == 228 + 28 * 2
    assert d["grid"] == 152
    assert d["launches"] == 1
    # per stage each CTA receives a 128x64 A box (16384 bytes, the pages'
    # transfer size of a 128x64 BF16 tile) and half the B rows
    assert d["stage_tx_bytes"] == 2 * (16384 + 128 * 64 * 2)
    assert d["smem_bytes"] <= 232448


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (4096, 14336, 4096), (3000, 5000, 2000),
                                   (8192, 8192, 8192), (512, 1000, 1000), (1000, 712, 136)])
def test_plan_pair_matches_wave_model(lib, M, N, K):
    st, p = _native.gemm_bf16_plan(M, N, K, _native.GEMM_OUT_F32, 152)
    d = p.as_dict()
    assert st == 0 and d["kernel_name"] == "pair"
    bn, split, units, _ = pair_model(M, N, K)
    assert (d["tile_n"], d["split_k"], d["tiles"]) == (bn, split, units)


def test_plan_pair_matches_wave_model_on_random_shapes(lib):
    """The planner against its restated wave model on seeded random shapes
    (M > 128, N and K up to 20000, FP32 and BF16 output)."""
    rng = np.random.default_rng(7)
    for _ in range(400):
        M = int(rng.integers(129, 20000))
        N, K = (int(x) for x in rng.integers(1, 20000, size=2))
        for od in (_native.GEMM_OUT_F32, _native.GEMM_OUT_BF16):
            st, p = _native.gemm_bf16_plan(M, N, K, od, 152)
            d = p.as_dict()
            assert st == 0 and d["kernel_name"] == "pair", (M, N, K)
            bn, split, units, _ = pair_model(M, N, K)
            assert (d["tile_n"], d["split_k"], d["tiles"]) == (bn, split, units), (M, N, K, od)


def test_plans_keep_their_invariants_on_random_shapes(lib):
    """Every plan over seeded random (batch, M, N, K), operand and output types
    fits the hardware and the kernels' fixed shapes: 1..232448 bytes of shared
    memory, 1..152 CTAs (an even number for CTA pairs), 64-element k-blocks,
    one launch; 256-row pair tiles, 128-row tiles elsewhere; the small-M
    activation tile the smallest of 16, 32, 64, 128 that holds M."""
    rng = np.random.default_rng(8)
    kinds = set()
    for _ in range(600):
        batch = int(rng.choice([1, 1, 1, int(rng.integers(2, 17))]))
        M = int(rng.choice([rng.integers(1, 17), rng.integers(17, 129), rng.integers(129, 8193)]))
        N, K = (int(x) for x in rng.integers(1, 20000, size=2))
        in_dtype, out_dtype = int(rng.integers(0, 2)), int(rng.integers(0, 3))
        st, p = _native.gemm_batched_plan(batch, M, N, K, in_dtype, out_dtype, 152)
        d = p.as_dict()
        case = (batch, M, N, K, in_dtype, out_dtype, d)
        assert st == 0, case
        assert 0 < d["smem_bytes"] <= 232448, case
        assert 1 <= d["grid"] <= 152, case
        assert d["split_k"] >= 1 and d["tiles"] >= 1, case
        assert d["tile_k"] == 64 and d["launches"] == 1, case
        k = d["kernel_name"]
        kinds.add(k)
        if k == "pair":
            assert d["grid"] % 2 == 0 and d["tile_m"] == 256 and d["tile_n"] in (224, 256), case
        else:
            assert d["tile_m"] == 128, case
        if k == "small_m":
            assert d["tile_n"] == min(n for n in (16, 32, 64, 128) if n >= M), case
        if k == "skinny_splitk":
            assert M <= 16 and d["tile_n"] == 16, case
    assert kinds == {"pair", "tiled", "skinny_splitk", "small_m"}


def test_plan_strips_cut_the_unsplit_tail_wave(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    # 3000 x 5000 x 2000: 12 x 20 = 240 tiles of 256 columns, 3 waves on 76
    # pairs and 12 left; 32 k-blocks cannot be cut into two pieces of 24, so
    # the 12 tiles run as 48 strips of 64 columns (3.63 waves x 576 against 4
    # waves of 224-wide tiles x 544)
    st, p = _native.gemm_bf16_plan(3000, 5000, 2000, _native.GEMM_OUT_F32, 152)
    assert st == 0
    assert (p.tile_n, p.split_k, p.tiles, p.grid) == (256, 1, 228 + 48, 152)
    monkeypatch.setenv("GB3_GEMM_STRIPS", "0")
    st, p = _native.gemm_bf16_plan(3000, 5000, 2000, _native.GEMM_OUT_F32, 152)
    assert (p.tile_n, p.split_k, p.tiles) == (224, 1, 276)
    # a tail that a K split serves keeps the split (4096^3: 28 tiles x 2 pieces)
    monkeypatch.delenv("GB3_GEMM_STRIPS")
    st, p = _native.gemm_bf16_plan(4096, 4096, 4096, _native.GEMM_OUT_BF16, 152)
    assert (p.tile_n, p.split_k, p.tiles) == (256, 2, 228 + 56)
    # forced: strips wherever the tail fits, also in place of a K split
    monkeypatch.setenv("GB3_GEMM_STRIPS", "1")
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", "256")
    st, p = _native.gemm_bf16_plan(2304, 4136, 4096, _native.GEMM_OUT_BF16, 152)
    assert (p.split_k, p.tiles) == (1, 153 - 1 + 4)
    # too many tail tiles for the pairs: 28 x 4 > 76
    st, p = _native.gemm_bf16_plan(4096, 4096, 2048, _native.GEMM_OUT_BF16, 152)
    assert (p.split_k, p.tiles) == (1, 256)


def test_plan_strips_not_with_row_stats(lib, monkeypatch):
    # the row-statistics kernels have no strip units: whole tiles only
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    st, p = _native.gemm_row_stats_plan(1, 3000, 5000, 2000, 0, _native.GEMM_OUT_F32, 152)
    assert st == 0 and (p.tile_n, p.tiles) == (224, 276)


def test_plan_balanced_after_whole_waves(lib, monkeypatch):
    """GB3_GEMM_BALANCED=2: all whole waves but the last run whole tiles, the
    rest of the tiles' k-blocks are divided into one range per pair."""
    monkeypatch.setenv("GB3_GEMM_BALANCED", "2")
    for M, N, K in [(4096, 4096, 4096), (8192, 8192, 8192), (2304, 4136, 200)]:
        st, p = _native.gemm_bf16_plan(M, N, K, _native.GEMM_OUT_F32, 152)
        assert st == 0 and p.tile_n in (256, 224)
        tiles = -(-M // 256) * -(-N // p.tile_n)
        dp = (tiles // 76 - 1) * 76
        units, pieces, _ = balanced_division(tiles - dp, -(-K // 64), 76)
        assert (p.tiles, p.split_k, p.grid) == (dp + units, pieces, 152)


def test_plan_tail_split_pieces_are_long_enough(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")   # the tail split alone
    # K = 2048 is 32 k-blocks: two pieces would be shorter than 24 k-blocks
    st, p = _native.gemm_bf16_plan(4096, 4096, 2048, _native.GEMM_OUT_BF16, 152)
    assert st == 0 and p.split_k == 1
    st, p = _native.gemm_bf16_plan(4096, 4096, 3072, _native.GEMM_OUT_BF16, 152)
    assert st == 0 and p.split_k == 2


def test_plan_forced_pair_width(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", "224")
    st, p = _native.gemm_bf16_plan(4096, 4096, 4096, _native.GEMM_OUT_BF16, 152)
    assert st == 0 and p.tile_n == 224 and p.tiles == 16 * 19 and p.split_k == 1
    monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", "100")   # not compiled: ignored
    st, p = _native.gemm_bf16_plan(4096, 4096, 4096, _native.GEMM_OUT_BF16, 152)
    assert st == 0 and p.tile_n == 256


def test_plan_split_overrides(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_TAIL_SPLIT", "0")
    monkeypatch.setenv("GB3_GEMM_BALANCED", "0")
    st, p = _native.gemm_bf16_plan(4096, 4096, 4096, _native.GEMM_OUT_BF16, 152)
    assert st == 0 and p.split_k == 1
    monkeypatch.setenv("GB3_GEMM_BALANCED", "1")
    st, p = _native.gemm_bf16_plan(4096, 4096, 4096, _native.GEMM_OUT_BF16, 152)
    assert st == 0 and p.split_k == 2 and p.tiles == balanced_division(256, 64, 76)[0]
    monkeypatch.delenv("GB3_GEMM_BALANCED")
    monkeypatch.delenv("GB3_GEMM_TAIL_SPLIT")
    monkeypatch.setenv("GB3_GEMM_SPLIT_ALL", "3")
    st, p = _native.gemm_bf16_plan(512, 1024, 1024, _native.GEMM_OUT_BF16, 152)
    assert st == 0 and p.split_k == 3
    tiles = 2 * -(-1024 // p.tile_n)
    assert p.tiles == tiles * 3


def test_plan_single_cta_below_two_row_blocks(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "0")
    st, p = _native.gemm_bf16_plan(128, 4096, 4096, _native.GEMM_OUT_BF16, 152)
    d = p.as_dict()
    assert st == 0 and d["kernel_name"] == "tiled"
    assert d["tile_m"] == 128 and d["tile_n"] == 256
    assert d["tiles"] == 16 and d["grid"] == 16
    assert d["stage_tx_bytes"] == 16384 + 256 * 64 * 2


def test_plan_ragged_tiles_cover_the_output(lib):
    st, p = _native.gemm_bf16_plan(3000, 5000, 2000, _native.GEMM_OUT_F32, 152)
    assert st == 0
    d = p.as_dict()
    tiles = -(-3000 // d["tile_m"]) * -(-5000 // d["tile_n"])
    # units: whole tiles plus the split pieces, or the four 64-column strips,
    # of the tail tiles; every tile is covered
    tail = tiles % 76
    if d["split_k"] > 1:
        assert d["tiles"] == tiles - tail + tail * d["split_k"]
    else:
        assert d["tile_n"] == 256 and d["tiles"] == tiles - tail + tail * 4


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (3000, 5000, 2000), (8192, 8192, 8192),
                                   (1000, 712, 136), (2304, 4136, 200)])
def test_plan_balanced_division_when_enabled(lib, monkeypatch, M, N, K):
    """GB3_GEMM_BALANCED=1: every pair takes one contiguous range of the tiles'
    k-blocks (where there are at least as many tiles as pairs)."""
    monkeypatch.setenv("GB3_GEMM_BALANCED", "1")
    st, p = _native.gemm_bf16_plan(M, N, K, _native.GEMM_OUT_F32, 152)
    d = p.as_dict()
    assert st == 0 and d["kernel_name"] == "pair"
    bn, split, units, balanced = pair_model(M, N, K, balanced=True)
    assert (d["tile_n"], d["split_k"], d["tiles"]) == (bn, split, units)
    tiles = -(-M // 256) * -(-N // bn)
    assert balanced == (tiles >= 76)
    if balanced:
        assert d["grid"] == 152


def test_plan_skinny_split_k(lib):
    st, p = _native.gemm_bf16_plan(16, 28672, 8192, _native.GEMM_OUT_BF16, 152)
    assert st == 0
    d = p.as_dict()
    assert d["kernel_name"] == "skinny_splitk"
    assert d["tile_m"] == 128 and d["tile_n"] == 16
    assert d["split_k"] == 2               # 224 row blocks alone: 1.5 waves
    kb = 8192 // 64
    kb_per = -(-kb // d["split_k"])
    assert -(-kb // kb_per) == d["split_k"]   # every split gets work
    assert d["tiles"] == 224 * d["split_k"]
    assert d["grid"] == 152
    # busiest CTA within 5% of a perfectly even spread of k-blocks
    busiest = -(-d["tiles"] // d["grid"]) * kb_per
    assert busiest <= 1.05 * (224 * kb) / 152
    assert d["stage_tx_bytes"] == 128 * 64 * 2 + 16 * 64 * 2


def test_plan_degenerate(lib):
    st, p = _native.gemm_bf16_plan(0, 10, 10, 1, 152)
    assert st == 0 and p.kernel == 0 and p.launches == 0
    st, p = _native.gemm_bf16_plan(10, 10, 0, 1, 152)
    assert st == 0 and p.as_dict()["kernel_name"] == "scale" and p.launches == 1
    assert _native.gemm_bf16_plan(-1, 10, 10, 1, 152)[0] == _native.GEMM_ERR_INVALID_ARG
    assert _native.gemm_bf16_plan(1, 10, 10, 5, 152)[0] == _native.GEMM_ERR_INVALID_ARG


def test_plan_gate_up(lib):
    st, p = _native.gemm_gate_up_plan(4096, 14336, 4096, 152)
    assert st == 0
    d = p.as_dict()
    assert d["kernel_name"] == "pair_gate_up"
    assert d["tile_m"] == 256 and d["tile_n"] == 128
    assert d["tiles"] == 16 * 112
    # per CTA: X box + (Wg box on the even CTA | Wu box on the odd CTA)
    assert d["stage_tx_bytes"] == 2 * 2 * 16384
    st, p = _native.gemm_gate_up_plan(100, 14336, 4096, 152)
    d = p.as_dict()
    assert d["kernel_name"] == "gate_up" and d["tile_m"] == 128
    assert d["stage_tx_bytes"] == 3 * 16384


def test_plan_gate_up_balanced_when_enabled(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_BALANCED", "1")
    st, p = _native.gemm_gate_up_plan(4096, 14336, 4096, 152)
    d = p.as_dict()
    units, pieces, _ = balanced_division(16 * 112, 64, 76)
    assert st == 0 and d["kernel_name"] == "pair_gate_up"
    assert d["tiles"] == units and d["split_k"] == pieces == 2


def test_plan_gate_up_decode(lib, monkeypatch):
    """M <= 16: Wg and Wu rows stream together through the split-K kernel."""
    for M in (1, 16):
        st, p = _native.gemm_gate_up_plan(M, 14336, 4096, 152)
        d = p.as_dict()
        assert st == 0 and d["kernel_name"] == "skinny_gate_up"
        assert d["tile_m"] == 128 and d["tile_n"] == 16
        assert d["stage_tx_bytes"] == 2 * 16384 + 2048      # Wg, Wu and X rows
        assert d["tiles"] == 112 * d["split_k"] and d["grid"] == min(d["tiles"], 152)
    st, p = _native.gemm_gate_up_plan(17, 14336, 4096, 152)
    assert p.as_dict()["kernel_name"] == "gate_up"
    monkeypatch.setenv("GB3_GATE_UP_SKINNY", "0")
    st, p = _native.gemm_gate_up_plan(16, 14336, 4096, 152)
    assert p.as_dict()["kernel_name"] == "gate_up"


def test_selftest_rejects_out_of_range_limits(lib):
    assert _native.gemm_selftest_wait_timeout(10, 0) == _native.GEMM_ERR_INVALID_ARG
    assert _native.gemm_selftest_wait_timeout(5 * 10**9, 0) == _native.GEMM_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# Row reductions, row normalisation and the normalised gate/up projection
# ---------------------------------------------------------------------------
F32, BF16, F16 = _native.GEMM_OUT_F32, _native.GEMM_OUT_BF16, _native.GEMM_OUT_F16


@pytest.mark.parametrize("args,expect", [
    # (rows, D, X, ldx, xk, G, eps, Y, ldy, yk)
    ((-1, 8, A16, 8, BF16, A16, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((8, -1, A16, 8, BF16, A16, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((1 << 31, 8, A16, 8, BF16, A16, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, A16, 8, 3, A16, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),   # x code
    ((8, 8, A16, 8, BF16, A16, 1e-6, A16 * 2, 8, 5), _native.GEMM_ERR_INVALID_ARG),   # y code
    ((8, 8, A16, 8, BF16, A16, -1.0, A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, A16, 8, BF16, A16, float("nan"), A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, A16, 8, BF16, A16, float("inf"), A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, 0, 8, BF16, A16, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),  # NULL X
    ((8, 8, A16, 8, BF16, 0, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_INVALID_ARG),  # NULL G
    ((8, 8, A16, 8, BF16, A16, 1e-6, 0, 8, BF16), _native.GEMM_ERR_INVALID_ARG),      # NULL Y
    ((8, 16, A16, 8, BF16, A16, 1e-6, A16 * 2, 16, BF16), _native.GEMM_ERR_INVALID_ARG),  # ldx<D
    ((8, 8, A16 + 2, 8, BF16, A16, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_ALIGNMENT),
    ((8, 8, A16, 8, BF16, A16 + 4, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_ALIGNMENT),
    ((8, 8, A16, 8, BF16, A16, 1e-6, A16 * 2 + 8, 8, BF16), _native.GEMM_ERR_ALIGNMENT),
    ((8, 4, A16, 4, BF16, A16, 1e-6, A16 * 2, 8, BF16), _native.GEMM_ERR_ALIGNMENT),  # ldx*2%16
    ((8, 6, A16, 8, F32, A16, 1e-6, A16 * 2, 6, F32), _native.GEMM_ERR_ALIGNMENT),    # ldy*4%16
    # Y overlapping X other than exactly in place
    ((8, 8, A16, 8, BF16, A16 * 3, 1e-6, A16 + 16, 8, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, A16, 8, F32, A16 * 3, 1e-6, A16, 8, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((8, 8, A16, 8, BF16, A16 * 3, 1e-6, A16, 16, BF16), _native.GEMM_ERR_INVALID_ARG),
    ((0, 8, 0, 8, BF16, 0, 1e-6, 0, 8, BF16), _native.GEMM_OK),                       # empty
    ((8, 0, 0, 0, BF16, 0, 0.0, 0, 0, BF16), _native.GEMM_OK),
])
def test_rms_norm_validation_without_gpu(lib, args, expect):
    assert _native.gemm_rms_norm(*args, 0) == expect


def test_rmsnorm_gate_up_validation_without_gpu(lib):
    ok = dict(M=8, N=8, K=8, X=A16, ldx=8, G=A16 * 3, eps=1e-6, Wg=A16 * 4, Wu=A16 * 5, ldw=8,
              Xn=A16 * 6, ldxn=8, Y=A16 * 7, ldy=8)

    def call(**kw):
        a = dict(ok, **kw)
        return _native.gemm_rmsnorm_gate_up_silu(a["M"], a["N"], a["K"], a["X"], a["ldx"],
                                                 a["G"], a["eps"], a["Wg"], a["Wu"], a["ldw"],
                                                 a["Xn"], a["ldxn"], a["Y"], a["ldy"], 0)
    assert call(M=-1) == _native.GEMM_ERR_INVALID_ARG
    assert call(eps=-1.0) == _native.GEMM_ERR_INVALID_ARG
    assert call(G=0) == _native.GEMM_ERR_INVALID_ARG
    assert call(Xn=0) == _native.GEMM_ERR_INVALID_ARG
    assert call(Xn=A16 + 16) == _native.GEMM_ERR_INVALID_ARG      # partly overlaps X
    assert call(G=A16 * 3 + 4) == _native.GEMM_ERR_ALIGNMENT
    assert call(Wg=A16 * 4 + 2) == _native.GEMM_ERR_ALIGNMENT
    assert call(ldxn=4) == _native.GEMM_ERR_INVALID_ARG
    assert call(M=0) == _native.GEMM_OK


def test_row_stats_validation_without_gpu(lib):
    def call(M=8, N=8, K=8, C=A16 * 2, rs=A16 * 3, rm=0, rn=0, in_dt=0, out_dt=BF16):
        return _native.gemm_row_stats(1, M, N, K, 1.0, A16, 8, 0, A16 * 4, 8, 0, 0.0, C, 8, 0,
                                      in_dt, out_dt, rs, rm, rn, 0)
    assert call(M=-1) == _native.GEMM_ERR_INVALID_ARG
    assert call(in_dt=2) == _native.GEMM_ERR_INVALID_ARG
    assert call(C=0) == _native.GEMM_ERR_INVALID_ARG
    assert call(rs=A16 * 3 + 2) == _native.GEMM_ERR_ALIGNMENT
    assert call(rm=A16 * 3 + 1) == _native.GEMM_ERR_ALIGNMENT
    assert call(M=0) == _native.GEMM_OK


def row_stats_plan(M, N, K, out=BF16):
    st, p = _native.gemm_row_stats_plan(1, M, N, K, 0, out, 148)
    assert st == _native.GEMM_OK
    return p.as_dict()


def test_row_stats_plans():
    # M <= 16 takes the 128-row tiled kernel instead of the swapped-operand one
    assert row_stats_plan(16, 4096, 4096)["kernel_name"] == "tiled"
    assert row_stats_plan(16, 28672, 8192)["kernel_name"] == "tiled"
    assert _native.gemm_batched_plan(1, 16, 28672, 8192, 0, BF16, 148)[1].as_dict()[
        "kernel_name"] == "skinny_splitk"
    # above M = 128 the same plan as the plain GEMM, except that the tail
    # wave is never cut into strips (the row-statistics kernels have none)
    for shape in [(300, 520, 200), (4096, 4096, 4096), (3000, 5000, 2000)]:
        a = row_stats_plan(*shape)
        b = _native.gemm_batched_plan(1, *shape, 0, BF16, 148)[1].as_dict()
        tiles = -(-shape[0] // 256) * -(-shape[1] // b["tile_n"])
        if b["tile_n"] == 256 and b["split_k"] == 1 and b["tiles"] > tiles:
            assert a["tiles"] == -(-shape[0] // 256) * -(-shape[1] // a["tile_n"])
        else:
            assert a == b
    # K == 0: the reductions of beta*C, then the scaling of C
    k0 = row_stats_plan(64, 64, 0)
    assert k0["kernel_name"] == "scale" and k0["launches"] == 2
    # N == 0: only the empty-row reductions
    n0 = row_stats_plan(64, 0, 64)
    assert n0["kernel_name"] == "scale" and n0["launches"] == 1


# ---------------------------------------------------------------------------
# The small-M kernel: 64-row weight tiles, k-block sequence divided evenly
# over the CTAs (stream-K)
# ---------------------------------------------------------------------------
def plan(M, N, K, batch=1, sms=152):
    st, p = _native.gemm_batched_plan(batch, M, N, K, 0, BF16, sms)
    assert st == _native.GEMM_OK
    return p.as_dict()


def test_plan_small_m_routing(lib):
    # 16 < M <= 128: 128-row weight tiles for at most every SM take the small-M kernel
    assert plan(64, 4096, 4096)["kernel_name"] == "small_m"          # 32 tiles
    assert plan(96, 8192, 8192)["kernel_name"] == "small_m"          # 64 tiles
    assert plan(128, 14336, 4096)["kernel_name"] == "small_m"        # 112 tiles
    assert plan(17, 19456, 4096)["kernel_name"] == "small_m"         # 152 tiles: one each
    assert plan(17, 19584, 4096)["kernel_name"] == "tiled"           # 153 tiles
    assert plan(64, 28672, 8192)["kernel_name"] == "tiled"           # 224 tiles
    # M <= 16: the small-M kernel while its tiles fill at most half the SMs
    assert plan(16, 8192, 8192)["kernel_name"] == "small_m"          # 64 tiles
    assert plan(1, 4096, 4096)["kernel_name"] == "small_m"           # 32 tiles
    assert plan(16, 9728, 4096)["kernel_name"] == "small_m"          # 76 tiles
    assert plan(16, 9856, 4096)["kernel_name"] == "skinny_splitk"    # 77 tiles
    assert plan(4, 14336, 8192)["kernel_name"] == "skinny_splitk"    # 112 tiles
    assert plan(16, 28672, 8192)["kernel_name"] == "skinny_splitk"   # 224 tiles
    assert plan(300, 4096, 4096)["kernel_name"] == "pair"            # M > 128
    import workloads
    w = workloads.WORKLOADS["smallm_64x8192x8192"]
    assert plan(w.M, w.N, w.K)["kernel_name"] == "small_m"


def test_plan_small_m_decode_shape(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "1")
    d = plan(64, 28672, 8192)
    # 224 tiles of 128 k-blocks on 152 CTAs: each CTA takes 188 or 189
    # k-blocks, so no tile is shared by more than two CTAs
    assert d["kernel_name"] == "small_m" and d["split_k"] == 2
    assert d["tile_m"] == 128 and d["tile_n"] == 64
    assert d["tiles"] == 28672 // 128 and d["grid"] == 152
    assert d["stage_tx_bytes"] == 128 * 64 * 2 + 64 * 64 * 2
    assert d["stages"] == 200 * 1024 // d["stage_tx_bytes"]
    assert d["smem_bytes"] <= 232448


@pytest.mark.parametrize("M,nx", [(1, 16), (16, 16), (17, 32), (32, 32), (33, 64), (64, 64),
                                  (65, 128), (128, 128)])
def test_plan_small_m_activation_tile(lib, monkeypatch, M, nx):
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "1")
    d = plan(M, 5000, 1000, batch=3)
    assert d["kernel_name"] == "small_m" and d["tile_n"] == nx
    assert d["tiles"] == 3 * -(-5000 // 128)


def _most_ctas_per_tile(tiles, k_blocks, grid):
    """Brute force: cut tiles * k_blocks positions into `grid` contiguous ranges
    whose lengths differ by at most one (the longer ones first) and count, for
    every tile, the ranges its positions fall in."""
    work = tiles * k_blocks
    owner = np.empty(work, dtype=np.int64)
    q, r = divmod(work, grid)
    pos = 0
    for c in range(grid):
        n = q + (1 if c < r else 0)
        owner[pos:pos + n] = c
        pos += n
    assert pos == work
    return max(len(set(owner[t * k_blocks:(t + 1) * k_blocks])) for t in range(tiles))


@pytest.mark.parametrize("batch,M,N,K,grid", [
    (1, 64, 8192, 8192, 152),    # 64 tiles x 128 k-blocks: divided over every SM
    (1, 64, 4096, 4096, 152),    # 32 tiles x 64
    (1, 16, 1000, 4096, 64),     # 8 tiles x 64: shares of 8 k-blocks
    (1, 128, 640, 1024, 10),     # 5 tiles x 16
    (3, 40, 200, 2048, 24),      # batched: ranges cross from one matrix to the next
    (1, 40, 1800, 8008, 152),    # ragged K
    (1, 33, 520, 200, 5),        # 4 k-blocks: one CTA per tile
    (1, 64, 9728, 4096, 152),    # 76 tiles: half the SMs, still divided
    (1, 64, 14336, 4096, 112),   # 112 tiles: one whole tile per CTA
    (1, 64, 28672, 8192, 152),   # 224 tiles: more than the SMs, divided
])
def test_plan_small_m_stream_k_division(lib, monkeypatch, batch, M, N, K, grid):
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "1")
    d = plan(M, N, K, batch=batch)
    tiles, kb = batch * -(-N // 128), -(-K // 64)
    assert d["kernel_name"] == "small_m" and d["tiles"] == tiles
    assert d["grid"] == grid
    assert d["split_k"] == _most_ctas_per_tile(tiles, kb, grid)


def test_plan_small_m_stream_k_switch(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "1")
    assert plan(64, 8192, 8192)["split_k"] > 1
    monkeypatch.setenv("GB3_SMALL_M_STREAM_K", "0")
    d = plan(64, 8192, 8192)
    assert d["grid"] == 64 and d["split_k"] == 1      # one CTA per whole tile
    monkeypatch.setenv("GB3_SMALL_M_STREAM_K", "1")
    d = plan(64, 14336, 4096)
    assert d["grid"] == 152 and d["split_k"] > 1      # divided although 112 tiles


def test_plan_small_m_limits(lib, monkeypatch):
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "1")
    assert plan(129, 28672, 8192)["kernel_name"] == "pair"      # above the widest tile
    assert plan(64, 28672, 0)["kernel_name"] == "scale"         # K == 0
    st, p = _native.gemm_row_stats_plan(1, 64, 28672, 8192, 0, BF16, 152)
    assert p.as_dict()["kernel_name"] == "tiled"                # row reductions need rows
    monkeypatch.setenv("GB3_GEMM_SMALL_M", "0")
    assert plan(64, 28672, 8192)["kernel_name"] == "tiled"
    assert plan(16, 28672, 8192)["kernel_name"] == "skinny_splitk"


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def attn(heads=2, Nq=256, Nk=256, D=128, scale=0.1, Q=A16, ldq=128, sq=256 * 128, K=A16 * 2,
         ldk=128, sk=256 * 128, V=A16 * 3, ldv=128, sv=256 * 128, O=A16 * 4, ldo=128,
         so=256 * 128, out=BF16):
    return _native.gemm_attention(heads, Nq, Nk, D, scale, Q, ldq, sq, K, ldk, sk, V, ldv, sv, O,
                                  ldo, so, out, 0)


@pytest.mark.parametrize("kw,expect", [
    (dict(heads=-1), _native.GEMM_ERR_INVALID_ARG),
    (dict(D=96), _native.GEMM_ERR_INVALID_ARG),                      # head dimension 64 or 128
    (dict(out=F16), _native.GEMM_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _native.GEMM_ERR_INVALID_ARG),
    (dict(scale=float("inf")), _native.GEMM_ERR_INVALID_ARG),
    (dict(Nk=0), _native.GEMM_ERR_INVALID_ARG),                      # no keys
    (dict(K=0), _native.GEMM_ERR_INVALID_ARG),
    (dict(ldv=64), _native.GEMM_ERR_INVALID_ARG),                    # pitch < D
    (dict(sq=255 * 128), _native.GEMM_ERR_INVALID_ARG),              # heads overlap
    (dict(V=A16 * 3 + 8), _native.GEMM_ERR_ALIGNMENT),
    (dict(heads=1, ldk=132), _native.GEMM_ERR_ALIGNMENT),
    (dict(heads=1, out=F32, ldo=130), _native.GEMM_ERR_ALIGNMENT),
    (dict(heads=0, Q=0, K=0, V=0, O=0), _native.GEMM_OK),            # empty: no-op
    (dict(Nq=0, Q=0, O=0), _native.GEMM_OK),
])
def test_attention_validation_without_gpu(lib, kw, expect):
    assert attn(**kw) == expect


def layout_smem(stages, stage_bytes, barriers, staging=0):
    """Dynamic shared memory of a kernel layout: 1024 bytes of alignment slack,
    the stage ring, the epilogue staging boxes, 8 bytes per mbarrier and 16
    bytes for the TMEM address and the abort flag."""
    return 1024 + stages * stage_bytes + staging + barriers * 8 + 16


@pytest.mark.parametrize("case", ["pair256", "pair224", "tiled", "skinny", "small_m16",
                                  "small_m64", "small_m128", "pair_gate_up", "gate_up",
                                  "skinny_gate_up"])
def test_plan_shared_memory_matches_kernel_layout(lib, monkeypatch, case):
    """The dynamic shared memory a plan reports (the size the library launches
    with) equals the layout its kernel indexes: A/B (or W/X) rows per stage,
    staging boxes of 4 KB (four epilogue warps x two), 2 * stages + 5 barriers.
    Every kernel also compares the size it was given with its layout at entry
    and records GEMM_ERR_CUDA (site 9) instead of running past its allocation."""
    kb = 64 * 2                                     # one 64-element BF16 row of a stage
    staging = 4 * 2 * 4096
    if case.startswith("pair2"):
        bn = int(case[4:])
        monkeypatch.setenv("GB3_GEMM_PAIR_TILE_N", str(bn))
        st, p = _native.gemm_bf16_plan(4096, 4096, 4096, _native.GEMM_OUT_BF16, 152)
        want = layout_smem(6, 128 * kb + bn // 2 * kb, 2 * 6 + 5, staging)
    elif case == "tiled":
        monkeypatch.setenv("GB3_GEMM_SMALL_M", "0")
        st, p = _native.gemm_bf16_plan(128, 4096, 4096, _native.GEMM_OUT_BF16, 152)
        want = layout_smem(4, 128 * kb + 256 * kb, 2 * 4 + 5, staging)
    elif case == "skinny":
        st, p = _native.gemm_bf16_plan(16, 28672, 8192, _native.GEMM_OUT_BF16, 152)
        want = layout_smem(12, 128 * kb + 16 * kb, 2 * 12 + 5)
    elif case.startswith("small_m"):
        nx = int(case[7:])
        st, p = _native.gemm_bf16_plan(nx, 8192, 8192, _native.GEMM_OUT_BF16, 152)
        stage = 128 * kb + nx * kb
        stages = (200 * 1024) // stage              # as many stages as fit in 200 KB
        want = layout_smem(stages, stage, 2 * stages + 5)
        assert p.stages == stages
    elif case == "pair_gate_up":
        st, p = _native.gemm_gate_up_plan(4096, 14336, 4096, 152)
        want = layout_smem(6, 128 * kb + 128 * kb, 2 * 6 + 5, staging)
    elif case == "gate_up":
        st, p = _native.gemm_gate_up_plan(100, 14336, 4096, 152)
        want = layout_smem(4, 128 * kb + 256 * kb, 2 * 4 + 5, staging)
    else:
        st, p = _native.gemm_gate_up_plan(16, 14336, 4096, 152)
        want = layout_smem(6, 2 * 128 * kb + 16 * kb, 2 * 6 + 5)
    assert st == 0
    assert p.smem_bytes == want and want <= 232448, (p.as_dict(), want)
