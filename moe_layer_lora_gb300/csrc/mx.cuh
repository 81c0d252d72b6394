// mx.cuh -- MXFP8 (OCP Microscaling Formats v1.0: blocks of 32 elements
// along the reduction dimension, one E8M0 scale 2^(s-127) per block, FP8
// E4M3 elements) for the layer's MXFP8 expert path, and the layout of the
// scale factors the tensor cores read.
//
// Conversion of a block, as the specification defines it: shared exponent
// = floor(log2(max |v|)) - 8 (8: the exponent of E4M3's largest normal,
// 448), clamped to >= -127 (a block of zeros or subnormals gets -127);
// element = v / 2^shared rounded to the nearest E4M3 value (ties to even)
// and saturated to +-448 -- one cvt.rn.satfinite.e4m3x2.f32 per pair.
#pragma once
#include <stdint.h>
#ifdef __CUDACC__
#include <cuda_bf16.h>
#endif

namespace mlora {

constexpr int kMxBlock = 32;       // elements per scale
constexpr int kMxChunk = 128;      // K per pipeline stage: one 128-byte swizzle row of E4M3
constexpr int kMxAtom = 512;       // scale bytes of 128 rows x one K-chunk (4 blocks)
constexpr int kMxWidth = 192;      // weight rows per MXFP8 tile (gate_up: 96 gate + 96 up)
constexpr int kMxHalf = kMxWidth / 2;
constexpr int kMxTileScaleBytes = 2 * kMxAtom;  // a tile's weight scales per K-chunk (rows 0-127, 128-191)

// Byte of row r (0..127) and K-block kb (0..3) inside a 512-byte atom.  The
// atom is 32 rows of 16 bytes: row r % 32 holds rows r, r+32, r+64, r+96,
// four bytes (one per K-block) each.  tcgen05.cp 32x128b.warpx4 puts it in
// tensor memory where the block-scaled MMA reads it: A row m at lane m,
// column m / 32; B row n at lane n % 32 (every lane quarter), column n / 32.
__host__ __device__ constexpr int mx_atom_byte(int r, int kb) { return (r % 32) * 16 + (r / 32) * 4 + kb; }

// Packed weight scales.  gate_up: for each expert e, tile slab cb of
// kMxHalf gate and kMxHalf up rows, K-chunk kc of H: kMxTileScaleBytes;
// tile row n < 96 is gate row cb*96 + n, n >= 96 up row I + cb*96 + n - 96.
// down: for each expert, slab cb of kMxWidth rows of w2, K-chunk kc of I.
__host__ __device__ constexpr long mx_slabs(int which, int H, int I) {
    return which == 0 ? (I + kMxHalf - 1) / kMxHalf : (H + kMxWidth - 1) / kMxWidth;
}
__host__ __device__ constexpr long mx_chunks(int which, int H, int I) {
    return which == 0 ? (H + kMxChunk - 1) / kMxChunk : (I + kMxChunk - 1) / kMxChunk;
}

#ifdef __CUDACC__
// Shared exponent of a block whose largest magnitude is amax (>= 0).
__device__ __forceinline__ int mx_shared_exp(float amax) {
    const int field = (__float_as_int(amax) >> 23) & 0xff;
    return field == 0 ? -127 : max(-127, field - 127 - 8);
}

// 2^-se exactly, for se in [-127, 119] (every finite fp32 block).
__device__ __forceinline__ float mx_inv_scale(int se) { return __int_as_float((127 - se) << 23); }

// Four values to four E4M3 codes, byte i = code of the i-th value.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    uint32_t lo, hi;
    asm("{.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;}" : "=r"(lo) : "f"(a), "f"(b));
    asm("{.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;}" : "=r"(hi) : "f"(c), "f"(d));
    return lo | (hi << 16);
}

// One block of 32 values (already in registers) to 32 codes (two uint4,
// bytes in element order) and its scale byte.
__device__ __forceinline__ uint8_t mx_quantize32(const float (&v)[32], uint4& q0, uint4& q1) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int se = mx_shared_exp(amax);
    const float inv = mx_inv_scale(se);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    q0 = make_uint4(w[0], w[1], w[2], w[3]);
    q1 = make_uint4(w[4], w[5], w[6], w[7]);
    return static_cast<uint8_t>(se + 127);
}

// One routed x row into sorted position p (row r = p % 128 of its block):
// each lane takes whole blocks of 32 of the bf16 row `src`, writes their
// E4M3 codes to q_row and their scale bytes into the block's atoms
// (atoms[kc * 512 + ...], kc = the K-chunk); the bf16 row is copied to
// bf_row too when it is set.  The loads of two blocks per lane are issued
// before either is converted; the four scale bytes of a K-chunk (lanes
// 4j..4j+3 of one pass) go out as one 32-bit word.  Blocks of the last
// K-chunk past H get a zero scale byte (their data reads as zero), never a
// stale one.  Every lane of the warp must call it.
__device__ __forceinline__ void mx_gather_row(const uint4* __restrict__ src, int H, int r, uint8_t* __restrict__ q_row,
                                              uint8_t* __restrict__ atoms, uint4* __restrict__ bf_row, int lane) {
    const int nblk = H / kMxBlock;
    const int nchunk = (H + kMxChunk - 1) / kMxChunk;
    const int passes = (nblk + 31) / 32;
    const int word_off = (r % 32) * 16 + (r / 32) * 4;  // the row's 4 scale bytes in an atom
    constexpr int kGroup = 2;
    for (int i0 = 0; i0 < passes; i0 += kGroup) {
        uint4 raw[kGroup][4];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int b = (i0 + u) * 32 + lane;
            if (i0 + u < passes && b < nblk) {
#pragma unroll
                for (int q = 0; q < 4; ++q) raw[u][q] = __ldg(src + b * 4 + q);
            }
        }
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            if (i0 + u >= passes) break;  // the same for every lane
            const int b = (i0 + u) * 32 + lane;
            uint32_t sc = 0;
            if (b < nblk) {
                if (bf_row) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) bf_row[b * 4 + q] = raw[u][q];
                }
                float v[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[u][q]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 t = __bfloat1622float2(h[i]);
                        v[8 * q + 2 * i] = t.x;
                        v[8 * q + 2 * i + 1] = t.y;
                    }
                }
                uint4 q0, q1;
                sc = mx_quantize32(v, q0, q1);
                uint4* dq = reinterpret_cast<uint4*>(q_row + b * kMxBlock);
                dq[0] = q0;
                dq[1] = q1;
            }
            uint32_t word = sc << (8 * (lane & 3));
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            const int kc = b / (kMxChunk / kMxBlock);
            if ((lane & 3) == 0 && kc < nchunk) *reinterpret_cast<uint32_t*>(atoms + kc * kMxAtom + word_off) = word;
        }
    }
}
#endif

}  // namespace mlora
