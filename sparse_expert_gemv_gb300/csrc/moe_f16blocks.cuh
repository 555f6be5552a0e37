// f16 block arithmetic shared by the kernels: activations (x, h) held in
// shared memory as 32-element blocks of f16, each block multiplied by the
// power of two 2^e that brings its largest magnitude into [2^14, 2^15) (the
// factor 2^-e is applied to the block's dot product), and weight codes
// converted to f16 with cvt.rn.f16x2.e4m3x2 (MXFP8) or cvt.rn.f16x2.e2m1x2
// (MXFP4). The two weight formats are the types Mxfp8 and Mxfp4 at the end,
// which every kernel takes as a template argument.
//
// Exactness: E4M3 -> f16 and E2M1 -> f16 are exact, a bf16 value scaled that
// way is exact in f16 whenever it lies within 2^-28 of its block's largest
// magnitude, and an f16 x f16 product is exact in FP32, so fma.rn.f32.f16
// gives the same sums as FP32 FMAs on the decoded values.
#pragma once

#include <cuda_fp16.h>

#include "moe_device.cuh"

namespace moe {

// Byte offset, inside a 64-byte block of 32 f16 values, of its 16-byte chunk c
// (values 8c .. 8c+7). Eight lanes reading eight consecutive blocks (a quarter
// warp, one shared-memory wavefront of 16-byte loads) ask for chunk 2f + i
// (i fixed, f = bit 2 of the block) in lanes with f = 0 and chunk 2(1 - f) + i
// in the others; XOR-ing the chunk index with bit 1 of the block then puts the
// eight loads in eight distinct 16-byte bank groups.
__device__ __forceinline__ int chunk_off(int block, int c) { return 16 * (c ^ ((block >> 1) & 1)); }

// 2^n as FP32 for -127 <= n <= 127, built from its bit pattern.
__device__ __forceinline__ float exp2i(int n) {
  return __uint_as_float(n > -127 ? (uint32_t)(n + 127) << 23 : 0x00400000u);
}

// One 32-element block of bf16 values (four uint4) -> f16 scaled by 2^e with
// the block's largest magnitude in [2^14, 2^15), written to a 64-byte block
// of shared memory; returns the factor 2^-e. A block of zeros (or of bf16
// subnormals only) takes e = 127; Inf and NaN stay Inf and NaN.
__device__ __forceinline__ float stage_block_f16(const uint4 (&v)[4], uint8_t* dst, int block) {
  uint32_t m = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t ww[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = max(m, max(ww[i] & 0x7fffu, (ww[i] >> 16) & 0x7fffu));
  }
  const int e = min(141 - (int)(m >> 7), 127);   // 14 - (biased exponent - 127)
  const float up = exp2i(e);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t ww[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 hh = __floats2half2_rn(bf16_lo(ww[i]) * up, bf16_hi(ww[i]) * up);
      o[i] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    *reinterpret_cast<uint4*>(dst + chunk_off(block, c)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  return exp2i(-e);
}

// Four E4M3 codes (one word, byte n = element n) times four f16 activations
// (two f16x2 words), added to two FP32 accumulators.
__device__ __forceinline__ void fma_e4m3x4(float& p, float& q, uint32_t codes, uint32_t x01,
                                           uint32_t x23) {
  asm("{\n\t.reg .b16 c0, c1;\n\t.reg .b32 lo, hi;\n\t"
      ".reg .f16 w0, w1, w2, w3, v0, v1, v2, v3;\n\t"
      "mov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 lo, c0;\n\tcvt.rn.f16x2.e4m3x2 hi, c1;\n\t"
      "mov.b32 {w0, w1}, lo;\n\tmov.b32 {w2, w3}, hi;\n\t"
      "mov.b32 {v0, v1}, %3;\n\tmov.b32 {v2, v3}, %4;\n\t"
      "fma.rn.f32.f16 %0, w0, v0, %0;\n\tfma.rn.f32.f16 %1, w1, v1, %1;\n\t"
      "fma.rn.f32.f16 %0, w2, v2, %0;\n\tfma.rn.f32.f16 %1, w3, v3, %1;\n\t}"
      : "+f"(p), "+f"(q)
      : "r"(codes), "r"(x01), "r"(x23));
}

// 16 codes (one uint4) against 16 f16 activations (two uint4).
__device__ __forceinline__ void fma_e4m3x16(float& p, float& q, const uint4 c, const uint4 x0,
                                            const uint4 x1) {
  fma_e4m3x4(p, q, c.x, x0.x, x0.y);
  fma_e4m3x4(p, q, c.y, x0.z, x0.w);
  fma_e4m3x4(p, q, c.z, x1.x, x1.y);
  fma_e4m3x4(p, q, c.w, x1.z, x1.w);
}

// A lane's view of one 32-element block: which 16-code half it reads first
// (alternating between groups of four lanes, so that a warp's 16-byte code
// loads at a 32-byte lane stride are free of bank conflicts) and the byte
// offsets of the matching activation chunks. Blocks a lane visits differ by
// multiples of 8, so this depends on the lane alone.
struct LaneBlock {
  int c_first, c_second;   // code half offsets (0 or 16)
  int x0, x1, x2, x3;      // activation chunk offsets for the first and second half
  __device__ __forceinline__ explicit LaneBlock(int lane) {
    const int f = (lane >> 2) & 1;
    c_first = 16 * f;
    c_second = 16 * (1 - f);
    x0 = chunk_off(lane, 2 * f);
    x1 = chunk_off(lane, 2 * f + 1);
    x2 = chunk_off(lane, 2 * (1 - f));
    x3 = chunk_off(lane, 2 * (1 - f) + 1);
  }
};

// Dot product of one block: 32 codes at `codes` (shared memory) against the
// f16 activation block at `act`.
__device__ __forceinline__ float dot_block(const uint8_t* codes, const uint8_t* act,
                                           const LaneBlock& lb) {
  const uint4 a = *reinterpret_cast<const uint4*>(codes + lb.c_first);
  const uint4 b = *reinterpret_cast<const uint4*>(codes + lb.c_second);
  const uint4 x0 = *reinterpret_cast<const uint4*>(act + lb.x0);
  const uint4 x1 = *reinterpret_cast<const uint4*>(act + lb.x1);
  const uint4 x2 = *reinterpret_cast<const uint4*>(act + lb.x2);
  const uint4 x3 = *reinterpret_cast<const uint4*>(act + lb.x3);
  float p = 0.f, q = 0.f, r = 0.f, s = 0.f;
  fma_e4m3x16(p, q, a, x0, x1);
  fma_e4m3x16(r, s, b, x2, x3);
  return (p + q) + (r + s);
}

// dot_block for two rows' codes (codes_a, codes_b) against one activation
// block, whose chunks are read once.
__device__ __forceinline__ void dot_block2(const uint8_t* codes_a, const uint8_t* codes_b,
                                           const uint8_t* act, const LaneBlock& lb, float& da,
                                           float& db) {
  const uint4 x0 = *reinterpret_cast<const uint4*>(act + lb.x0);
  const uint4 x1 = *reinterpret_cast<const uint4*>(act + lb.x1);
  const uint4 x2 = *reinterpret_cast<const uint4*>(act + lb.x2);
  const uint4 x3 = *reinterpret_cast<const uint4*>(act + lb.x3);
  const uint4 a0 = *reinterpret_cast<const uint4*>(codes_a + lb.c_first);
  const uint4 a1 = *reinterpret_cast<const uint4*>(codes_a + lb.c_second);
  const uint4 b0 = *reinterpret_cast<const uint4*>(codes_b + lb.c_first);
  const uint4 b1 = *reinterpret_cast<const uint4*>(codes_b + lb.c_second);
  float p = 0.f, q = 0.f, r = 0.f, s = 0.f;
  fma_e4m3x16(p, q, a0, x0, x1);
  fma_e4m3x16(r, s, a1, x2, x3);
  da = (p + q) + (r + s);
  p = q = r = s = 0.f;
  fma_e4m3x16(p, q, b0, x0, x1);
  fma_e4m3x16(r, s, b1, x2, x3);
  db = (p + q) + (r + s);
}

// Four E4M3 codes (one word) -> two f16x2 words: elements 0,1 and 2,3.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t codes, uint32_t& w01, uint32_t& w23) {
  asm("{\n\t.reg .b16 c0, c1;\n\tmov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c0;\n\tcvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
      : "=r"(w01), "=r"(w23)
      : "r"(codes));
}

// Four products of f16 pairs (weights w01, w23 against activations x01, x23)
// added to two FP32 accumulators.
__device__ __forceinline__ void fma_f16x4(float& p, float& q, uint32_t w01, uint32_t w23,
                                          uint32_t x01, uint32_t x23) {
  asm("{\n\t.reg .f16 w0, w1, w2, w3, v0, v1, v2, v3;\n\t"
      "mov.b32 {w0, w1}, %2;\n\tmov.b32 {w2, w3}, %3;\n\t"
      "mov.b32 {v0, v1}, %4;\n\tmov.b32 {v2, v3}, %5;\n\t"
      "fma.rn.f32.f16 %0, w0, v0, %0;\n\tfma.rn.f32.f16 %1, w1, v1, %1;\n\t"
      "fma.rn.f32.f16 %0, w2, v2, %0;\n\tfma.rn.f32.f16 %1, w3, v3, %1;\n\t}"
      : "+f"(p), "+f"(q)
      : "r"(w01), "r"(w23), "r"(x01), "r"(x23));
}

// One weight block (32 codes in q, this lane's half first when LaneBlock says
// so) decoded to 16 f16x2 words in that order.
__device__ __forceinline__ void decode_block_f16(const uint32_t (&q)[8], bool swap,
                                                 uint32_t (&wh)[16]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t v = swap ? q[c ^ 4] : q[c];
    e4m3x4_to_f16x2(v, wh[2 * c], wh[2 * c + 1]);
  }
}

// The block dot of decoded weights against the f16 activation block at act.
__device__ __forceinline__ float dot_block_h(const uint32_t (&wh)[16], const uint8_t* act,
                                             const LaneBlock& lb) {
  const uint4 x0 = *reinterpret_cast<const uint4*>(act + lb.x0);
  const uint4 x1 = *reinterpret_cast<const uint4*>(act + lb.x1);
  const uint4 x2 = *reinterpret_cast<const uint4*>(act + lb.x2);
  const uint4 x3 = *reinterpret_cast<const uint4*>(act + lb.x3);
  float p = 0.f, q = 0.f, r = 0.f, s = 0.f;
  fma_f16x4(p, q, wh[0], wh[1], x0.x, x0.y);
  fma_f16x4(p, q, wh[2], wh[3], x0.z, x0.w);
  fma_f16x4(p, q, wh[4], wh[5], x1.x, x1.y);
  fma_f16x4(p, q, wh[6], wh[7], x1.z, x1.w);
  fma_f16x4(r, s, wh[8], wh[9], x2.x, x2.y);
  fma_f16x4(r, s, wh[10], wh[11], x2.z, x2.w);
  fma_f16x4(r, s, wh[12], wh[13], x3.x, x3.y);
  fma_f16x4(r, s, wh[14], wh[15], x3.z, x3.w);
  return (p + q) + (r + s);
}

// dot_block_h with the activation chunks already in registers (x0 .. x3 as
// LaneBlock orders them: x0, x1 with wh[0..7], x2, x3 with wh[8..15]).
__device__ __forceinline__ float dot_regs16(const uint32_t (&wh)[16], const uint4& x0,
                                            const uint4& x1, const uint4& x2, const uint4& x3) {
  float p = 0.f, q = 0.f, r = 0.f, s = 0.f;
  fma_f16x4(p, q, wh[0], wh[1], x0.x, x0.y);
  fma_f16x4(p, q, wh[2], wh[3], x0.z, x0.w);
  fma_f16x4(p, q, wh[4], wh[5], x1.x, x1.y);
  fma_f16x4(p, q, wh[6], wh[7], x1.z, x1.w);
  fma_f16x4(r, s, wh[8], wh[9], x2.x, x2.y);
  fma_f16x4(r, s, wh[10], wh[11], x2.z, x2.w);
  fma_f16x4(r, s, wh[12], wh[13], x3.x, x3.y);
  fma_f16x4(r, s, wh[14], wh[15], x3.z, x3.w);
  return (p + q) + (r + s);
}

// ---------------------------------------------------------------------------
// MXFP4 elements: E2M1 codes, two to a byte, element 2c in the low nibble of
// byte c (the element format the GC-MoE summary, onedev.kr/papers/1690, "How
// it is used", gives its routed weights; the packing follows the OCP MX
// convention). cvt.rn.f16x2.e2m1x2 turns one byte into an f16 pair, its low
// nibble into the low half.
// ---------------------------------------------------------------------------

// Eight E2M1 codes (one word, nibble n = element n) -> four f16x2 words:
// elements 0,1 / 2,3 / 4,5 / 6,7.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t codes, uint32_t& w01, uint32_t& w23,
                                                uint32_t& w45, uint32_t& w67) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(w01), "=r"(w23), "=r"(w45), "=r"(w67)
      : "r"(codes));
}

// f16x2 word -> two FP32 values (exact).
__device__ __forceinline__ void f16x2_to_f32(uint32_t w, float& lo, float& hi) {
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w));
}

// ---------------------------------------------------------------------------
// The weight formats. Each describes one 32-element block of a weight row:
//   kBlockBytes    code bytes of the block (rows are K * kBlockBytes / 32 bytes)
//   kWords         32-bit words holding them
//   load(p, q)     the block's codes from global memory (streamed, see ld_weights32)
//   decode(q, swap, wh)  16 f16x2 words: elements 0..15 then 16..31, or the
//                  two halves the other way round when `swap` (the order in
//                  which LaneBlock pairs them with activation chunks)
//   chunk_f32(q, c, v)   elements 8c .. 8c+7 as FP32
//   dot_smem(codes, act, lb)  the block's dot with an f16 activation block,
//                  codes read from shared memory
//   kLaneBytes, lds_lane(p, w), decode_lane(w, f)  one lane's eight
//                  consecutive codes of a block (the tensor-core fragment
//                  layout of moe_gate_up_tma: kLaneBytes bytes in kLaneWords
//                  words, read from shared memory) and their four f16x2 pairs
// ---------------------------------------------------------------------------

struct Mxfp8 {
  static constexpr int kBlockBytes = 32;
  static constexpr int kWords = 8;
  __device__ __forceinline__ static void load(const uint8_t* p, uint32_t (&q)[kWords]) {
    ld_weights32(p, q);
  }
  __device__ __forceinline__ static void decode(const uint32_t (&q)[kWords], bool swap,
                                                uint32_t (&wh)[16]) {
    decode_block_f16(q, swap, wh);
  }
  __device__ __forceinline__ static void chunk_f32(const uint32_t (&q)[kWords], int c,
                                                   float (&v)[8]) {
    e4m3x4_to_f32(q[2 * c], v[0], v[1], v[2], v[3]);
    e4m3x4_to_f32(q[2 * c + 1], v[4], v[5], v[6], v[7]);
  }
  __device__ __forceinline__ static float dot_smem(const uint8_t* codes, const uint8_t* act,
                                                   const LaneBlock& lb) {
    return dot_block(codes, act, lb);
  }
  __device__ __forceinline__ static void dot2_smem(const uint8_t* codes_a, const uint8_t* codes_b,
                                                   const uint8_t* act, const LaneBlock& lb,
                                                   float& da, float& db) {
    dot_block2(codes_a, codes_b, act, lb, da, db);
  }
  static constexpr int kLaneBytes = 8;
  static constexpr int kLaneWords = 2;
  __device__ __forceinline__ static void lds_lane(const uint8_t* p, uint32_t (&w)[kLaneWords]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x;
    w[1] = v.y;
  }
  __device__ __forceinline__ static void decode_lane(const uint32_t (&w)[kLaneWords],
                                                     uint32_t (&f)[4]) {
    e4m3x4_to_f16x2(w[0], f[0], f[1]);
    e4m3x4_to_f16x2(w[1], f[2], f[3]);
  }
};

struct Mxfp4 {
  static constexpr int kBlockBytes = 16;
  static constexpr int kWords = 4;
  __device__ __forceinline__ static void load(const uint8_t* p, uint32_t (&q)[kWords]) {
    ld_weights16(p, q);
  }
  __device__ __forceinline__ static void decode(const uint32_t (&q)[kWords], bool swap,
                                                uint32_t (&wh)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t v = swap ? q[c ^ 2] : q[c];
      e2m1x8_to_f16x2(v, wh[4 * c], wh[4 * c + 1], wh[4 * c + 2], wh[4 * c + 3]);
    }
  }
  __device__ __forceinline__ static void chunk_f32(const uint32_t (&q)[kWords], int c,
                                                   float (&v)[8]) {
    uint32_t w[4];
    e2m1x8_to_f16x2(q[c], w[0], w[1], w[2], w[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) f16x2_to_f32(w[i], v[2 * i], v[2 * i + 1]);
  }
  // A warp's 32 lanes read 32 consecutive 16-byte blocks: conflict-free
  // without the half swap MXFP8's 32-byte blocks need, so the codes are
  // reordered in registers instead.
  __device__ __forceinline__ static float dot_smem(const uint8_t* codes, const uint8_t* act,
                                                   const LaneBlock& lb) {
    const uint4 a = *reinterpret_cast<const uint4*>(codes);
    const uint32_t q[4] = {a.x, a.y, a.z, a.w};
    uint32_t wh[16];
    decode(q, lb.c_first != 0, wh);
    return dot_block_h(wh, act, lb);
  }
  __device__ __forceinline__ static void dot2_smem(const uint8_t* codes_a, const uint8_t* codes_b,
                                                   const uint8_t* act, const LaneBlock& lb,
                                                   float& da, float& db) {
    const uint4 x0 = *reinterpret_cast<const uint4*>(act + lb.x0);
    const uint4 x1 = *reinterpret_cast<const uint4*>(act + lb.x1);
    const uint4 x2 = *reinterpret_cast<const uint4*>(act + lb.x2);
    const uint4 x3 = *reinterpret_cast<const uint4*>(act + lb.x3);
    const uint4 a = *reinterpret_cast<const uint4*>(codes_a);
    const uint4 b = *reinterpret_cast<const uint4*>(codes_b);
    const uint32_t qa[4] = {a.x, a.y, a.z, a.w}, qb[4] = {b.x, b.y, b.z, b.w};
    uint32_t wh[16];
    decode(qa, lb.c_first != 0, wh);
    da = dot_regs16(wh, x0, x1, x2, x3);
    decode(qb, lb.c_first != 0, wh);
    db = dot_regs16(wh, x0, x1, x2, x3);
  }
  static constexpr int kLaneBytes = 4;
  static constexpr int kLaneWords = 1;
  __device__ __forceinline__ static void lds_lane(const uint8_t* p, uint32_t (&w)[kLaneWords]) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
  __device__ __forceinline__ static void decode_lane(const uint32_t (&w)[kLaneWords],
                                                     uint32_t (&f)[4]) {
    e2m1x8_to_f16x2(w[0], f[0], f[1], f[2], f[3]);
  }
};

}  // namespace moe
