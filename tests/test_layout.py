"""The encodings the kernels compute, checked field by field on the CPU through
the library's host-only layout calls (the same functions the kernels call):
the 128-byte swizzle of operand tiles and staging boxes, Tensor Memory
addresses, the shared-memory matrix descriptor and the tcgen05 instruction
descriptor.  A wrong bit in any of them would otherwise show only as a wrong
result, or a fault, on the GPU.

Worked values from the pages: element (1, 0) of a 128-byte-swizzled tile of
16-bit elements sits at element offset 72 and a 128 x 64 BF16 box transfers
16384 bytes ("TMA and Hopper WGMMA", section "The same storage contract on
both sides"); Tensor Memory lane 64, column 32 is address (64 << 16) + 32
("TMEM tiles and transfers", section "Storage and a transfer").  The
descriptor bit fields follow the PTX ISA's tcgen05 descriptor tables.
"""
import pytest

from dense_bf16_gemm_gb300 import _native


@pytest.fixture(scope="module")
def lib():
    return _native.lib()


def bits(v, lo, hi):
    """Bits lo..hi (inclusive) of v."""
    return (v >> lo) & ((1 << (hi - lo + 1)) - 1)


def element_offset(lib, r, k):
    """Element offset of (row r, K index k) in a swizzled tile of 16-bit elements."""
    byte = lib.gemm_layout_swizzle128_offset(r, k // 8) + (k % 8) * 2
    assert byte % 2 == 0
    return byte // 2


def test_swizzle_worked_value(lib):
    assert element_offset(lib, 1, 0) == 72
    assert element_offset(lib, 0, 0) == 0


def test_swizzle_matches_the_pages_formula_on_every_element(lib):
    # 64 r + (k xor 8 (r mod 8)) for every element of a 32-row box and of a
    # 128-row operand tile (the swizzle phase repeats every 8 rows)
    for r in range(128):
        for k in range(64):
            assert element_offset(lib, r, k) == 64 * r + (k ^ (8 * (r % 8))), (r, k)


def test_swizzle_is_a_permutation_of_each_row(lib):
    for r in range(16):
        offs = sorted(element_offset(lib, r, k) for k in range(64))
        assert offs == list(range(64 * r, 64 * r + 64))


def test_box_transfer_bytes(lib):
    # a 128 x 64 BF16 box is 16384 bytes: the A share of every pipeline stage
    st, p = _native.gemm_bf16_plan(4096, 4096, 4096, _native.GEMM_OUT_BF16, 152)
    assert st == 0
    assert 128 * 64 * 2 == 16384
    assert p.stage_tx_bytes == 2 * (16384 + (p.tile_n // 2) * 64 * 2)


def test_tmem_address_worked_value(lib):
    assert lib.gemm_layout_tmem_address(0, 64, 32) == (64 << 16) + 32
    # lanes in bits 31:16, columns in bits 15:0, added to the allocation's base
    base = 256
    for lane in (0, 32, 96, 127):
        for col in (0, 31, 255, 511):
            a = lib.gemm_layout_tmem_address(base, lane, col)
            assert a == base + (lane << 16) + col
            assert bits(a, 16, 31) == lane and bits(a, 0, 15) == base + col


@pytest.mark.parametrize("addr", [0, 1024, 17408, 99328, 230400])
def test_k_major_smem_descriptor_fields(lib, addr):
    d = lib.gemm_layout_smem_descriptor(addr, 0)
    assert bits(d, 0, 13) == (addr & 0x3FFFF) >> 4      # start address >> 4
    assert bits(d, 16, 29) == 1                         # leading offset: unused, 1
    assert bits(d, 32, 45) == 1024 >> 4                 # 8-row groups 1024 bytes apart
    assert bits(d, 46, 47) == 1                         # descriptor version
    assert bits(d, 49, 51) == 0                         # base offset: 1024-aligned tiles
    assert bits(d, 52, 52) == 0                         # relative leading-offset mode
    assert bits(d, 61, 63) == 2                         # 128-byte swizzle
    used = (0x3FFF | (0x3FFF << 16) | (0x3FFF << 32) | (3 << 46) | (7 << 49) | (1 << 52)
            | (7 << 61))
    assert d & ~used & (2 ** 64 - 1) == 0               # nothing else set


def test_k_major_descriptor_steps_along_k(lib):
    # the kernels advance an operand by one K = 16 step (32 bytes of a
    # 128-byte row) by adding 2 to the descriptor
    for base in (0, 1024, 65536):
        d0 = lib.gemm_layout_smem_descriptor(base, 0)
        for j in range(4):
            assert lib.gemm_layout_smem_descriptor(base + 32 * j, 0) == d0 + 2 * j


@pytest.mark.parametrize("chunk", [16384, 32768])
def test_mn_major_smem_descriptor_fields(lib, chunk):
    d = lib.gemm_layout_smem_descriptor(2048, chunk)
    assert bits(d, 0, 13) == 2048 >> 4
    assert bits(d, 16, 29) == chunk >> 4                # 64-element MN chunks apart
    assert bits(d, 32, 45) == 1024 >> 4
    assert bits(d, 46, 47) == 1
    assert bits(d, 61, 63) == 2


@pytest.mark.parametrize("M,N", [(128, 256), (256, 256), (256, 224), (128, 64), (128, 16),
                                 (64, 64), (128, 128)])
@pytest.mark.parametrize("in_dtype", [_native.GEMM_IN_BF16, _native.GEMM_IN_F16])
def test_instruction_descriptor_fields(lib, M, N, in_dtype):
    d = lib.gemm_layout_instr_descriptor(M, N, in_dtype)
    fmt = 1 if in_dtype == _native.GEMM_IN_BF16 else 0
    assert bits(d, 0, 3) == 0            # dense, no saturation
    assert bits(d, 4, 5) == 1            # D is FP32
    assert bits(d, 6, 6) == 0
    assert bits(d, 7, 9) == fmt          # A: BF16 = 1, FP16 = 0
    assert bits(d, 10, 12) == fmt        # B: the same type as A
    assert bits(d, 13, 14) == 0          # no negation
    assert bits(d, 15, 16) == 0          # A and B K-major
    assert bits(d, 17, 22) == N >> 3
    assert bits(d, 23, 23) == 0
    assert bits(d, 24, 28) == M >> 4
    assert bits(d, 29, 31) == 0          # no shift of D


def test_layout_calls_are_exported(lib):
    for name in ("gemm_layout_smem_descriptor", "gemm_layout_instr_descriptor",
                 "gemm_layout_swizzle128_offset", "gemm_layout_tmem_address"):
        assert name in _native.EXPORTED and hasattr(lib, name)


def test_descriptors_step_by_adding_to_the_start_field(lib):
    # the attention kernel steps its descriptors instead of re-encoding them:
    # 16 rows of an MN-major operand (2048 bytes) add 128, a 64-element chunk
    # of 128 K-major rows (16384 bytes) adds 1024, a K = 16 step adds 2
    for base in (1024, 17408, 98304, 200704):
        for kk in range(8):
            assert (lib.gemm_layout_smem_descriptor(base + kk * 2048, 16384)
                    == lib.gemm_layout_smem_descriptor(base, 16384) + 128 * kk)
        for ch in range(2):
            for kk in range(4):
                assert (lib.gemm_layout_smem_descriptor(base + ch * 16384 + 32 * kk, 0)
                        == lib.gemm_layout_smem_descriptor(base, 0) + 1024 * ch + 2 * kk)
