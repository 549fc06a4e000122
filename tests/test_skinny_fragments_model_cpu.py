"""The few-token kernel's 32-K operand loads, modelled on the CPU.

With 1-byte codes and up to 8 tokens (and E4M3 with two token groups), the
weight-streaming kernel (csrc/skinny.cuh) feeds `mma.sync m16n8k32`: int8 x
int8 -> int32, or E4M3 x E4M3 -> fp32.  Compute warp w owns the 32-K block w
of every 256-K stage.  Within a 128-byte swizzled box that is 16-byte chunks
c0 = 2 (w % 4) and c0 + 1 of every row, where logical chunk c of row r sits
at physical chunk c ^ (r & 7).

The operands come in through `ldmatrix` (m8n8, b16 elements):
  * lane l gives the address of row l % 8 of matrix l / 8;
  * every lane t receives the 4 bytes 4 (t % 4) .. + 4 of row t / 4 of each
    matrix.

The m16n8k32 fragments (PTX ISA, 8-bit operands), with g = lane / 4 and
q = lane % 4:
  * A: a0 = A[g][4q..4q+3], a1 = A[g+8][4q..4q+3], a2 = A[g][16+4q..],
    a3 = A[g+8][16+4q..];
  * B: b0 = B[4q..4q+3][g], b1 = B[16+4q..][g] (B stored token-major, so
    token g's codes 4q..4q+3).

This model computes the kernel's addresses for every warp, weight tile and
token group, reads a box filled with distinct byte labels through them, and
checks two things: the registers hold exactly those fragments, and each
8-lane address group is served in one wavefront (no bank conflicts).  It
also counts the 64-bit per-lane loads kept for E4M3 with one token group:
every half-warp puts two rows on the same banks, so they take twice the
minimum wavefronts.
"""
import os

ROWS = 64


def phys(row, chunk):
    """Byte offset in a 128-byte-swizzled box of logical (row, 16-byte chunk)."""
    return row * 128 + ((chunk ^ (row & 7)) << 4)


def box_bytes(rows, seed):
    """A box image holding, for every logical (row, k), the label (row, k)."""
    img = {}
    for r in range(rows):
        for k in range(128):
            img[phys(r, k // 16) + k % 16] = (seed, r, k)
    return img


def ldmatrix(img, addrs, nmat):
    """Registers of every lane for ldmatrix.x{nmat}: lane t gets bytes
    4 (t % 4) .. + 4 of row t / 4 of each matrix; matrix i's row j is at the
    address given by lane 8 i + j."""
    regs = []
    for t in range(32):
        out = []
        for i in range(nmat):
            base = addrs[8 * i + t // 4]
            out.append(tuple(img[base + 4 * (t % 4) + b] for b in range(4)))
        regs.append(out)
    return regs


def a_off(lane, w):
    li = lane & 7
    c0 = 2 * (w & 3)
    return (li + 8 * ((lane >> 3) & 1)) * 128 + (((c0 + (lane >> 4)) ^ li) << 4)


def b_off(lane, w):
    li = lane & 7
    c0 = 2 * (w & 3)
    return li * 128 + (((c0 + ((lane >> 3) & 1)) ^ li) << 4)


def wavefronts_per_group(addrs, width):
    """Wavefronts of one shared access whose lanes each read `width` bytes,
    served in groups of 128 bytes' worth of lanes: the most distinct words
    any bank sees within a group."""
    per = 128 // width
    total = 0
    for g0 in range(0, len(addrs), per):
        banks = {}
        for a in addrs[g0:g0 + per]:
            assert a % width == 0
            for wd in range(width // 4):
                word = a // 4 + wd
                banks.setdefault(word % 32, set()).add(word)
        total += max(len(v) for v in banks.values())
    return total


def test_ldmatrix_gives_the_m16n8k32_fragments():
    n = 0
    for w in range(8):
        kb = 32 * (w & 3)               # the block's first K within its box (w / 4)
        wimg = box_bytes(ROWS, "w")
        for rt in range(4):
            regs = ldmatrix(wimg, [16 * rt * 128 + a_off(l, w) for l in range(32)], 4)
            for lane in range(32):
                g, q = lane >> 2, lane & 3
                want = [
                    tuple(("w", 16 * rt + g, kb + 4 * q + b) for b in range(4)),
                    tuple(("w", 16 * rt + g + 8, kb + 4 * q + b) for b in range(4)),
                    tuple(("w", 16 * rt + g, kb + 16 + 4 * q + b) for b in range(4)),
                    tuple(("w", 16 * rt + g + 8, kb + 16 + 4 * q + b) for b in range(4)),
                ]
                assert regs[lane] == want, (w, rt, lane)
                n += 1
        for mt in (1, 2):
            timg = box_bytes(8 * mt, "x")
            for t in range(mt):
                regs = ldmatrix(timg, [8 * t * 128 + b_off(l, w) for l in range(32)], 2)
                for lane in range(32):
                    g, q = lane >> 2, lane & 3
                    want = [tuple(("x", 8 * t + g, kb + 4 * q + b) for b in range(4)),
                            tuple(("x", 8 * t + g, kb + 16 + 4 * q + b) for b in range(4))]
                    assert regs[lane] == want, (w, mt, t, lane)
    assert n == 8 * 4 * 32


def test_ldmatrix_addresses_are_conflict_free():
    for w in range(8):
        for rt in range(4):
            addrs = [16 * rt * 128 + a_off(l, w) for l in range(32)]
            # each 8-lane group is one matrix: eight 16-byte rows, one wavefront
            assert wavefronts_per_group(addrs, 16) == 4, (w, rt)
        for t in range(2):
            addrs = [8 * t * 128 + b_off(l, w) for l in range(16)]
            assert wavefronts_per_group(addrs, 16) == 2, (w, t)


def test_per_lane_64_bit_loads_conflict_two_ways():
    """The E4M3 one-group path keeps 64-bit per-lane loads: lane (g, q) reads
    8 bytes of row g at chunk (c0 + q / 2) ^ g.  Rows g and g ^ 1 land on the
    same 32 bytes of banks, so each half-warp takes two wavefronts, four per
    access instead of two."""
    for w in range(8):
        c0 = 2 * (w & 3)
        for rt in range(4):
            for hi in (0, 8):
                addrs = []
                for lane in range(32):
                    g, q = lane >> 2, lane & 3
                    off = (((c0 + (q >> 1)) ^ g) << 4) | (8 * (q & 1))
                    addrs.append((16 * rt + g + hi) * 128 + off)
                assert wavefronts_per_group(addrs, 8) == 4, (w, rt, hi)


def test_model_restates_the_kernel_source():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "w8a8_int8_quantized_i8_gb300", "csrc", "skinny.cuh")
    src = " ".join(open(path).read().split())
    for frag in (
        "const uint32_t c0 = 2u * static_cast<uint32_t>(w & 3);",
        "const uint32_t li = static_cast<uint32_t>(lane & 7);",
        "const uint32_t a_off = (li + 8u * static_cast<uint32_t>((lane >> 3) & 1)) * 128u + "
        "(((c0 + static_cast<uint32_t>(lane >> 4)) ^ li) << 4);",
        "const uint32_t b_off = li * 128u + (((c0 + static_cast<uint32_t>((lane >> 3) & 1)) ^ li) << 4);",
        "ldsm_x4(wbox + static_cast<uint32_t>(16 * rt) * 128u + a_off, wa[rt][0], wa[rt][1], wa[rt][2], wa[rt][3]);",
        "ldsm_x2(abox + static_cast<uint32_t>(8 * t) * 128u + b_off, xb[t][0], xb[t][1]);",
        "const uint32_t wbox = st + static_cast<uint32_t>((w >> 2) * Cfg::W_BOX_BYTES);",
        "mma_m16n8k32_s8(acc[rt][t], wa[rt][0], wa[rt][1], wa[rt][2], wa[rt][3], xb[t][0], xb[t][1]);",
        "static constexpr bool LDSM = K32 && !(FP8 && MT == 1);",
    ):
        assert frag in src, frag
