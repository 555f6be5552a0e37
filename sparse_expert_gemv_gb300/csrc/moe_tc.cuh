// Expert-centric tensor-core form of the decode layer, for batches too large
// for output-centric warp decode to win (the warp-decode post, "Warp decode
// and Composer training": prefill and large batches still favour packing
// tokens per expert). It is the operand-swapped Blackwell MMA the GC-MoE
// summary (onedev.kr/papers/1690), "How it is used", describes for its
// grouped GEMM: weight rows are the MMA's M dimension and the tokens routed to
// an expert are its N dimension, so a handful of tokens still fills the
// 128-row tensor-core tile.
//
// Four launches per group of up to 256 tokens:
//   moe_tc_prep      the unique experts, each expert's (token, slot) pairs in
//                    ascending slot order, their column chunks of <= 64 pairs,
//                    and x gathered into expert order (xg[p] = x[token of p])
//   moe_tc_gate_up   per tile (chunk, 128 neurons): gate and up rows decoded
//                    from MXFP8/MXFP4 to exact bf16 into tensor memory (the
//                    MMA's A operand), xg rows by TMA into shared memory (B),
//                    tcgen05.mma kind::f16 with FP32 accumulators in tensor
//                    memory; epilogue h = SiLU(g) * u -> bf16 into hg (expert
//                    order) and the caller's h[t, j]
//   moe_tc_down      per tile (chunk, 128 rows of y): W_down rows decoded the
//                    same way against hg; epilogue writes each pair's FP32
//                    partial row yp[p]
//   moe_tc_combine   y[t] = bf16(sum_j topk_w[t, j] * yp[pair of (t, j)]), in
//                    slot order (deterministic, no atomics)
//
// Exactness: an MX weight is code * 2^(s - 127). E4M3 and E2M1 codes convert
// exactly to f16 (always normal there), and the f16 -> bf16 move below keeps
// every bit, so with the scale folded in, the decoded weight is the exact
// value whenever it is a normal bf16: scale codes 10..142 (MXFP8) or 2..142
// (MXFP4), with no E4M3 NaN code. The host checks this once per handle and
// uses the path only then. x is bf16 already; bf16 x bf16 products are exact
// in the FP32 accumulator.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "moe_device.cuh"
#include "moe_f16blocks.cuh"

namespace moe {

constexpr int kTcMaxTokens = 256;   // tokens per group (pairs <= 256 * k)
constexpr int kTcRows = 128;        // weight rows per MMA (M)
constexpr int kTcCols = 64;         // pairs per column chunk (MMA N <= 64)
constexpr int kTcK = 64;            // K elements per pipeline stage
constexpr int kTcBBox = 16;         // rows per TMA box of the B operand
constexpr int kTcSB = 4;            // B-operand ring slots
constexpr int kTcGuSA = 4;          // tensor-memory A stages, gate/up
constexpr int kTcDnSA = 8;          // tensor-memory A stages, down
constexpr int kTcNS = 2;            // gate/up scale-chunk slots
constexpr int kTcScaleStages = 8;   // stages per gate/up scale chunk (16 scale bytes a row)
constexpr int kTcFirstDecodeWarp = 7;
constexpr int kTcGuDecodeWarps = 16;
constexpr int kTcDnDecodeWarps = 8;
constexpr int kTcGuThreads = (kTcFirstDecodeWarp + kTcGuDecodeWarps) * 32;
// gate/up decode warps: one per (lane quarter, tensor-memory A stage)
static_assert(kTcGuDecodeWarps == 4 * kTcGuSA && (kTcGuSA & (kTcGuSA - 1)) == 0, "decode warps");
// stage lanes split every scale chunk evenly
static_assert(kTcScaleStages % kTcGuSA == 0, "scale chunk");
constexpr int kTcDnThreads = (kTcFirstDecodeWarp + kTcDnDecodeWarps) * 32;
// down decode warps: four lane quarters x kTcDnLanes stage lanes
constexpr int kTcDnLanes = kTcDnDecodeWarps / 4;
static_assert(kTcDnLanes == 2 && kTcDnSA % kTcDnLanes == 0, "down decode warps");
constexpr int kTcPrepThreads = 512;
constexpr int kTcCombineThreads = 256;
// warp roles (both projection kernels)
constexpr int kTcWarpRaw = 0;       // weight codes (and scales) by TMA
constexpr int kTcWarpMma = 1;       // tensor-memory owner and MMA issuer
constexpr int kTcWarpB = 2;         // B operand by TMA
constexpr int kTcWarpEpi = 3;       // warps 3..6: epilogue, one per lane quarter
// tensor-memory columns: gate/up accumulators 2 x (64 gate + 64 up), then
// 4 A stages of 64 (32 gate + 32 up); down accumulators 2 x 64, then 8 A
// stages of 32
constexpr uint32_t kTcTmemCols = 512;
constexpr uint32_t kTcGuAcol = 256;
constexpr uint32_t kTcDnAcol = 128;
// scale codes for which every decoded weight is a normal bf16
constexpr int kTcScaleMinFp8 = 10;
constexpr int kTcScaleMinFp4 = 2;
constexpr int kTcScaleMax = 142;
// gate/up scale codes for which every decoded weight is exact in f16 (E4M3
// values are multiples of 2^-9 below 448, E2M1 values multiples of 2^-1 up
// to 6; f16 holds multiples of 2^-24 below 65520, and the scale 2^(s-127)
// itself is a normal f16 from s = 113)
constexpr int kTcF16ScaleMin = 113;
constexpr int kTcF16ScaleMaxFp8 = 134;
constexpr int kTcF16ScaleMaxFp4 = 140;

// Device views of the path's workspace (sized for kTcMaxTokens * k pairs).
struct TcWork {
  int* hdr;          // [0] pairs nP, [1] unique experts nU, [2] column chunks nC
  int* chunk_e;      // expert id of chunk c
  int* chunk_p0;     // its first pair (row of xg, hg and yp)
  int* chunk_n;      // its pairs, 1..kTcCols
  int* pair_slot;    // slot t*k + j of pair p
  int* slot_pair;    // pair of slot t*k + j, -1 for an id outside [0, E)
  uint16_t* xg;      // [pairs, H] bf16: x of each pair's token
  uint16_t* hg;      // [pairs, I] bf16: h of each pair
  float* yp;         // [pairs, H] FP32: W_down[e] h of each pair
  float* xinv;       // [pairs] with an f16 xg: 2^-e of the pair's token's row
};

struct TcPrepParams {
  const uint16_t* x;
  const int32_t* ids;
  uint16_t* h;       // caller's h: slots with invalid ids are zeroed here
  uint32_t* err;
  TcWork w;
  int T, k, E, H, I;
  // 0: xg holds x as is (bf16); 1: each row scaled by the power of two 2^e
  // that brings its token's largest magnitude into [2^14, 2^15), in f16,
  // with 2^-e in w.xinv
  int f16;
};

struct TcParams {
  CUtensorMap tm_w;  // weight codes: uint8 [rows, row bytes], boxes of 128 rows x one stage
  CUtensorMap tm_s;  // gate/up scales: uint8 [rows, H/32], boxes of 128 rows x 16
  CUtensorMap tm_b;  // B operand: bf16 [pairs, K], boxes of 16 rows x 64, 128-byte swizzle
  const uint8_t* sd; // W_down scales (whole tiles by bulk copy)
  uint16_t* h;       // caller's h [T, k, I]
  uint32_t* err;
  TcWork w;
  int E, H, I;
  int R;             // weight-code ring slots
};

struct TcCombineParams {
  const float* tw;   // topk_w [T, k]
  uint16_t* y;       // [T, H]
  TcWork w;
  int T, k, H;
};

// ---------------------------------------------------------------------------
// tcgen05 (tensor memory, MMA) and TMA wrappers
// ---------------------------------------------------------------------------
namespace tc {

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (both operands bf16 here).
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier when every MMA this thread issued so far is done.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Instruction descriptor of kind::f16: FP32 D, bf16 A and B (f16 A and B
// when !bf16), both K-major, M = 128, N = n (a multiple of 16, 16..256).
__device__ __forceinline__ uint32_t idesc_m128(int n, bool bf16) {
  return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(kTcRows >> 4) << 24);
}

// Shared-memory descriptor of a K-major operand written with the 128-byte
// swizzle (rows of 128 bytes, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// 16 consecutive 32-bit columns of this warp's 32 lanes <-> 16 registers.
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}

// ---------------------------------------------------------------------------
// MX -> bf16 decode of one 32-element block (one scale)
// ---------------------------------------------------------------------------

// bf16 pair (2^(s-15), 2^(s-15)), for scale codes 0 < s + 112 < 255.
__device__ __forceinline__ uint32_t scale_pair(uint32_t s) {
  return ((s + 112u) << 7) * 0x00010001u;
}

// An f16 pair whose values are normal or zero and whose low three mantissa
// bits are zero (any E4M3 or E2M1 value) -> the bf16 pair of the same values
// times 2^-112: each half's exponent and mantissa move down three bits into
// the wider bf16 exponent field, the sign stays. Then times 2^(s-15) (f2),
// exact while the product is a normal bf16: the weight code * 2^(s-127).
__device__ __forceinline__ uint32_t f16x2_to_scaled_bf16x2(uint32_t h, uint32_t f2) {
  const uint32_t t = ((h & 0x7FFF7FFFu) >> 3) | (h & 0x80008000u);
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(f2));
  return r;
}

// 32 E4M3 codes (byte n of the 8 words = element n) -> 16 bf16 pairs.
__device__ __forceinline__ void decode_fp8_block(const uint4& a, const uint4& b, uint32_t s,
                                                 uint32_t (&o)[16]) {
  const uint32_t f2 = scale_pair(s);
  const uint32_t q[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 u, v;\n\tmov.b32 {u, v}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, u;\n\tcvt.rn.f16x2.e4m3x2 %1, v;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(q[i]));
    o[2 * i] = f16x2_to_scaled_bf16x2(lo, f2);
    o[2 * i + 1] = f16x2_to_scaled_bf16x2(hi, f2);
  }
}

// 32 E2M1 codes (16 bytes; element 2c in the low nibble of byte c) -> 16
// bf16 pairs.
__device__ __forceinline__ void decode_fp4_block(const uint4& a, uint32_t s, uint32_t (&o)[16]) {
  const uint32_t f2 = scale_pair(s);
  const uint32_t q[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t w0, w1, w2, w3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
        : "r"(q[i]));
    o[4 * i] = f16x2_to_scaled_bf16x2(w0, f2);
    o[4 * i + 1] = f16x2_to_scaled_bf16x2(w1, f2);
    o[4 * i + 2] = f16x2_to_scaled_bf16x2(w2, f2);
    o[4 * i + 3] = f16x2_to_scaled_bf16x2(w3, f2);
  }
}

// f16 pair (2^(s-127), 2^(s-127)), for scale codes 113 <= s <= 142.
__device__ __forceinline__ uint32_t scale_pair_f16(uint32_t s) {
  return ((s - 112u) << 10) * 0x00010001u;
}

// 32 E4M3 codes -> 16 f16 pairs of code * 2^(s-127): the conversion, then one
// f16 multiply a pair (exact for the scale codes kTcF16ScaleMin ..
// kTcF16ScaleMaxFp8).
__device__ __forceinline__ void decode_fp8_block_f16(const uint4& a, const uint4& b, uint32_t s,
                                                     uint32_t (&o)[16]) {
  const uint32_t f2 = scale_pair_f16(s);
  const uint32_t q[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 u, v;\n\tmov.b32 {u, v}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, u;\n\tcvt.rn.f16x2.e4m3x2 %1, v;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(q[i]));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * i]) : "r"(lo), "r"(f2));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * i + 1]) : "r"(hi), "r"(f2));
  }
}

// 32 E2M1 codes -> 16 f16 pairs of code * 2^(s-127) (exact for the scale
// codes kTcF16ScaleMin .. kTcF16ScaleMaxFp4).
__device__ __forceinline__ void decode_fp4_block_f16(const uint4& a, uint32_t s,
                                                     uint32_t (&o)[16]) {
  const uint32_t f2 = scale_pair_f16(s);
  const uint32_t q[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t w[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
        : "r"(q[i]));
#pragma unroll
    for (int j = 0; j < 4; ++j) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[4 * i + j]) : "r"(w[j]), "r"(f2));
  }
}

}  // namespace tc

// The two weight formats as the tensor-core kernels read them: code bytes of
// a row per 64-element stage (the TMA swizzle they land with follows from
// it), the load of this thread's 32-element half of row r from a landed
// stage, and its decode.
struct TcFp8 {
  static constexpr int kStageRowBytes = 64;   // 64-byte swizzle: chunk c at c ^ ((r >> 1) & 3)
  __device__ __forceinline__ static void load(const uint8_t* rows, int r, int half,
                                              uint4 (&c)[2]) {
    const uint8_t* row = rows + r * kStageRowBytes;
    const int x = (r >> 1) & 3;
    c[0] = *reinterpret_cast<const uint4*>(row + 16 * ((2 * half) ^ x));
    c[1] = *reinterpret_cast<const uint4*>(row + 16 * ((2 * half + 1) ^ x));
  }
  __device__ __forceinline__ static void decode(const uint4 (&c)[2], uint32_t s,
                                                uint32_t (&o)[16]) {
    tc::decode_fp8_block(c[0], c[1], s, o);
  }
  __device__ __forceinline__ static void decode_f16(const uint4 (&c)[2], uint32_t s,
                                                    uint32_t (&o)[16]) {
    tc::decode_fp8_block_f16(c[0], c[1], s, o);
  }
};
struct TcFp4 {
  static constexpr int kStageRowBytes = 32;   // 32-byte swizzle: chunk c at c ^ ((r >> 2) & 1)
  __device__ __forceinline__ static void load(const uint8_t* rows, int r, int half,
                                              uint4 (&c)[2]) {
    const uint8_t* row = rows + r * kStageRowBytes;
    c[0] = *reinterpret_cast<const uint4*>(row + 16 * (half ^ ((r >> 2) & 1)));
    c[1] = c[0];
  }
  __device__ __forceinline__ static void decode(const uint4 (&c)[2], uint32_t s,
                                                uint32_t (&o)[16]) {
    tc::decode_fp4_block(c[0], s, o);
  }
  __device__ __forceinline__ static void decode_f16(const uint4 (&c)[2], uint32_t s,
                                                    uint32_t (&o)[16]) {
    tc::decode_fp4_block_f16(c[0], s, o);
  }
};

// ---------------------------------------------------------------------------
// moe_tc_prep: the dedup schedule of a token group (rows A1 of the layer's
// schedule: unique experts ascending, each expert's pairs in ascending slot
// order) and the gather of x into expert order. Every CTA builds the
// schedule in shared memory (at most 256 * 32 ids), so each can gather its
// rows at once; CTA 0 also publishes it.
// Dynamic shared memory: (3 * T * k + (16 + 3) * E) ints.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTcPrepThreads, 1) moe_tc_prep(const __grid_constant__ TcPrepParams p) {
  extern __shared__ int sm[];
  constexpr int NW = kTcPrepThreads / 32;
  const int P = p.T * p.k, E = p.E;
  int* sid = sm;            // id of slot i, -1 when outside [0, E)
  int* spos = sid + P;      // pair of slot i
  int* pslot = spos + P;    // slot of pair q
  int* cw = pslot + P;      // [NW][E]: a warp's count, then its offset within the expert
  int* cnt = cw + NW * E;   // pairs of expert e
  int* off = cnt + E;       // first pair of expert e
  int* cb = off + E;        // first column chunk of expert e
  __shared__ int s_tot[3];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ids and x come from upstream work, and the workspace is free once the
  // previous launch on the stream has finished
  pdl_wait();
  pdl_trigger();
  for (int i = tid; i < NW * E; i += kTcPrepThreads) cw[i] = 0;
  int bad = 0;
  for (int i = tid; i < P; i += kTcPrepThreads) {
    const int v = __ldg(p.ids + i);
    const bool ok = v >= 0 && v < E;
    sid[i] = ok ? v : -1;
    bad |= ok ? 0 : 1;
  }
  bad = __syncthreads_or(bad);

  // each warp counts its contiguous slice of slots, 32 at a time; lanes with
  // equal ids find each other and the highest adds their number
  const int slice = (P + NW - 1) / NW;
  const int s0 = min(P, warp * slice), s1 = min(P, s0 + slice);
  for (int b = s0; b < s1; b += 32) {
    const int i = b + lane;
    const int e = i < s1 ? sid[i] : -1;
    const uint32_t peers = __match_any_sync(kFull, e);
    if (e >= 0 && lane == 31 - __clz(peers)) cw[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = tid; e < E; e += kTcPrepThreads) {
    int run = 0;
    for (int w = 0; w < NW; ++w) {
      const int c = cw[w * E + e];
      cw[w * E + e] = run;
      run += c;
    }
    cnt[e] = run;
  }
  __syncthreads();
  // exclusive prefix sums over the experts of their pairs and chunks
  if (warp == 0) {
    int run_p = 0, run_c = 0, nu = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? cnt[e] : 0;
      const int nc = (c + kTcCols - 1) / kTcCols;
      int ip = c, ic = nc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(kFull, ip, o), b = __shfl_up_sync(kFull, ic, o);
        if (lane >= o) {
          ip += a;
          ic += b;
        }
      }
      if (e < E) {
        off[e] = run_p + ip - c;
        cb[e] = run_c + ic - nc;
      }
      nu += __popc(__ballot_sync(kFull, c > 0));
      run_p += __shfl_sync(kFull, ip, 31);
      run_c += __shfl_sync(kFull, ic, 31);
    }
    if (lane == 0) {
      s_tot[0] = run_p;
      s_tot[1] = nu;
      s_tot[2] = run_c;
    }
  }
  __syncthreads();
  // pair of each slot: the expert's first pair, plus the slots of the same
  // expert in earlier warps' slices, earlier batches and lower lanes
  for (int b = s0; b < s1; b += 32) {
    const int i = b + lane;
    const int e = i < s1 ? sid[i] : -1;
    const uint32_t peers = __match_any_sync(kFull, e);
    const int pos = e >= 0 ? off[e] + cw[warp * E + e] + __popc(peers & ((1u << lane) - 1u)) : -1;
    __syncwarp();
    if (e >= 0 && lane == 31 - __clz(peers)) cw[warp * E + e] += __popc(peers);
    if (i < s1) {
      spos[i] = pos;
      if (pos >= 0) pslot[pos] = i;
    }
    __syncwarp();
  }
  __syncthreads();
  const int nP = s_tot[0];
  if (blockIdx.x == 0) {
    if (tid == 0) {
      p.w.hdr[0] = nP;
      p.w.hdr[1] = s_tot[1];
      p.w.hdr[2] = s_tot[2];
      if (bad) atomicOr(p.err, kDeviceBadId);
    }
    for (int i = tid; i < P; i += kTcPrepThreads) p.w.slot_pair[i] = spos[i];
    for (int q = tid; q < nP; q += kTcPrepThreads) p.w.pair_slot[q] = pslot[q];
    for (int e = tid; e < E; e += kTcPrepThreads) {
      const int c = cnt[e];
      for (int j = 0; j * kTcCols < c; ++j) {
        p.w.chunk_e[cb[e] + j] = e;
        p.w.chunk_p0[cb[e] + j] = off[e] + j * kTcCols;
        p.w.chunk_n[cb[e] + j] = min(kTcCols, c - j * kTcCols);
      }
    }
  }
  // xg[q] = x[token of pair q] for pairs q = blockIdx.x, + gridDim.x, ...
  const int vpr = p.H / 8;   // 16-byte vectors a row
  const int rows = nP > (int)blockIdx.x ? (nP - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (p.f16) {
    // one warp a row: the token's largest magnitude, then the row in f16
    // times the power of two 2^e that brings it into [2^14, 2^15) (as the
    // warp kernels stage x, over the whole row here), and 2^-e
    for (int r = warp; r < rows; r += NW) {
      const int q = blockIdx.x + r * gridDim.x;
      const int t = pslot[q] / p.k;
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H);
      uint32_t m = 0;
      for (int c = lane; c < vpr; c += 32) {
        const uint4 v = __ldg(src + c);
        const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) m = max(m, max(ww[i] & 0x7fffu, (ww[i] >> 16) & 0x7fffu));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
      const int e = min(141 - (int)(m >> 7), 127);
      const float up = exp2i(e);
      for (int c = lane; c < vpr; c += 32) {
        const uint4 v = __ldg(src + c);
        const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
        uint32_t o4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 hh = __floats2half2_rn(bf16_lo(ww[i]) * up, bf16_hi(ww[i]) * up);
          o4[i] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        reinterpret_cast<uint4*>(p.w.xg + (size_t)q * p.H)[c] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      if (lane == 0) p.w.xinv[q] = exp2i(-e);
    }
  } else {
    for (int v = tid; v < rows * vpr; v += kTcPrepThreads) {
      const int q = blockIdx.x + (v / vpr) * gridDim.x, c = v % vpr;
      const int t = pslot[q] / p.k;
      reinterpret_cast<uint4*>(p.w.xg + (size_t)q * p.H)[c] =
          __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H) + c);
    }
  }
  // the caller's h slices of slots with invalid ids are zero
  if (bad) {
    const int vh = p.I / 8;
    for (int i = blockIdx.x; i < P; i += gridDim.x) {
      if (spos[i] >= 0) continue;
      for (int c = tid; c < vh; c += kTcPrepThreads)
        reinterpret_cast<uint4*>(p.h + (size_t)i * p.I)[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Shared memory of moe_tc_prep for P = T * k slots.
__host__ __device__ constexpr size_t tc_prep_smem(int P, int E) {
  return (size_t)(3 * P + (kTcPrepThreads / 32 + 3) * E) * sizeof(int);
}

// ---------------------------------------------------------------------------
// The projection kernels' shared-memory carve-up (1024-byte aligned pieces:
// the 128-byte swizzle repeats every 1024 bytes).
// ---------------------------------------------------------------------------
struct TcSmem {
  int raw, rawStage, b, sc, scStage, bars, total;
  // gate/up (down = false): raw stages of gate then up rows, the B ring, the
  // scale-chunk ring; down: raw stages of 128 rows, the B ring, two tiles of
  // scales (128 rows of I/32 bytes)
  __host__ __device__ TcSmem(bool down, int stageRowBytes, int R, int I) {
    rawStage = (down ? 1 : 2) * kTcRows * stageRowBytes;
    raw = 0;
    b = raw + R * rawStage;
    scStage = down ? (kTcRows * (I / 32) + 1023) / 1024 * 1024 : 2 * kTcRows * 16;
    sc = b + kTcSB * kTcCols * 128;
    bars = sc + (down ? 2 : kTcNS) * scStage;
    total = bars + (2 * R + 2 * kTcSB + 2 * kTcDnSA + 2 * kTcNS + 16) * 8 + 16;
  }
};

// Bounded wait on an mbarrier phase; a timeout marks the CTA dead (every
// role then winds down) and sets kDeviceTimeout.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                        volatile int* dead) {
  if (*dead) return false;
  if (mbar_wait(bar, parity, err)) return true;
  *dead = 1;
  return false;
}
// The same for a whole warp: true only when every lane saw the phase.
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity, uint32_t* err,
                                             volatile int* dead) {
  const bool ok = tc_wait(bar, parity, err, dead);
  return __all_sync(kFull, ok);
}

// ---------------------------------------------------------------------------
// moe_tc_gate_up: one persistent CTA per SM over tiles (chunk c, neurons
// [128 m, 128 m + 128)). Per 64-element stage of H: the raw-code warp brings
// the tile's 128 gate rows and 128 up rows by TMA (and every 8 stages their
// 16 scale bytes a row), 16 decode warps turn them into exact f16 or bf16 in
// tensor memory (warp quarter q owns lanes 32q..32q+31 = rows; the four
// warps of a quarter take every fourth stage, gate and up, so four stages
// are in decode at once), the B warp brings the chunk's xg rows, and one thread
// issues 2 x 4 MMAs (gate and up, K = 16 each) into the tile's accumulators.
// Four epilogue warps turn a finished tile into h while the next one runs.
// ---------------------------------------------------------------------------
// F16: the weights decode to f16 (scale codes in kTcF16ScaleMin ..
// kTcF16ScaleMax*) against xg in f16 (per-token power-of-two scaling, undone
// by w.xinv in the epilogue), else to bf16 against xg in bf16.
template <class F, bool F16>
__global__ void __launch_bounds__(kTcGuThreads, 1) moe_tc_gate_up(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int RB = F::kStageRowBytes;
  const int R = p.R;
  const TcSmem L(false, RB, R, p.I);
  uint8_t* raw = smem + L.raw;
  uint8_t* bbuf = smem + L.b;
  uint8_t* sc = smem + L.sc;
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* raw_empty = raw_full + R;
  uint64_t* b_full = raw_empty + R;
  uint64_t* b_empty = b_full + kTcSB;
  uint64_t* a_full = b_empty + kTcSB;
  uint64_t* a_empty = a_full + kTcGuSA;
  uint64_t* sc_full = a_empty + kTcGuSA;
  uint64_t* sc_empty = sc_full + kTcNS;
  uint64_t* d_full = sc_empty + kTcNS;
  uint64_t* d_empty = d_full + 2;
  uint64_t* drain = d_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* dead = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, I = p.I;
  const int nS = H / kTcK;          // stages a tile
  const int MT = I / kTcRows;       // neuron tiles an expert

  if (warp == kTcWarpRaw && lane == 0) {
    tc::prefetch_tmap(&p.tm_w);
    tc::prefetch_tmap(&p.tm_s);
  }
  if (warp == kTcWarpB && lane == 0) tc::prefetch_tmap(&p.tm_b);
  if (warp == kTcWarpEpi && lane == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], 4);   // the four lane quarters' decode warps of the stage
    }
    for (int i = 0; i < kTcSB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kTcGuSA; ++i) {
      mbar_init(&a_full[i], 4);      // the four lane quarters' decode warps of the slot
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kTcNS; ++i) {
      mbar_init(&sc_full[i], 1);
      mbar_init(&sc_empty[i], kTcGuDecodeWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 4);
    }
    mbar_init(drain, 1);
    *dead = 0;
    mbar_init_fence();
  }
  if (warp == kTcWarpMma) tc::tmem_alloc(tmem_slot, kTcTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // the schedule and xg come from moe_tc_prep
  const int ntiles = p.w.hdr[2] * MT;

  if (warp == kTcWarpRaw) {
    if (lane == 0) {
      int gs = 0, gc = 0;
      RingPos rw(R);   // the raw ring's slot and phase (no division by R per stage)
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
        const int c = tile / MT, m = tile % MT;
        const int rg = p.w.chunk_e[c] * 2 * I + m * kTcRows;   // gate rows; up rows I further
        for (int s = 0; ok && s < nS; ++s, ++gs) {
          if (s % kTcScaleStages == 0) {
            const int slot = gc % kTcNS;
            if (gc >= kTcNS) ok = tc_wait(&sc_empty[slot], ((gc / kTcNS) - 1) & 1, p.err, dead);
            if (!ok) break;
            uint8_t* dst = sc + slot * L.scStage;
            mbar_expect_tx(&sc_full[slot], L.scStage);
            tma_load_2d(dst, &p.tm_s, (s / kTcScaleStages) * 16, rg, &sc_full[slot]);
            tma_load_2d(dst + kTcRows * 16, &p.tm_s, (s / kTcScaleStages) * 16, rg + I, &sc_full[slot]);
            ++gc;
          }
          const int slot = rw.slot;
          if (gs >= R) ok = tc_wait(&raw_empty[slot], rw.phase ^ 1u, p.err, dead);
          if (!ok) break;
          uint8_t* dst = raw + slot * L.rawStage;
          mbar_expect_tx(&raw_full[slot], L.rawStage);
          tma_load_2d(dst, &p.tm_w, s * RB, rg, &raw_full[slot]);
          tma_load_2d(dst + kTcRows * RB, &p.tm_w, s * RB, rg + I, &raw_full[slot]);
          rw.next();
        }
      }
      // never leave with copies in flight
      for (int d = gs - R < 0 ? 0 : gs - R; d < gs; ++d) mbar_wait(&raw_full[d % R], (d / R) & 1, p.err);
      for (int d = gc - kTcNS < 0 ? 0 : gc - kTcNS; d < gc; ++d)
        mbar_wait(&sc_full[d % kTcNS], (d / kTcNS) & 1, p.err);
    }
  } else if (warp == kTcWarpB) {
    if (lane == 0) {
      int gs = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
        const int c = tile / MT;
        const int p0 = p.w.chunk_p0[c], nb = (p.w.chunk_n[c] + kTcBBox - 1) / kTcBBox;
        for (int s = 0; s < nS; ++s, ++gs) {
          const int slot = gs % kTcSB;
          if (gs >= kTcSB) ok = tc_wait(&b_empty[slot], ((gs / kTcSB) - 1) & 1, p.err, dead);
          if (!ok) break;
          uint8_t* dst = bbuf + slot * (kTcCols * 128);
          mbar_expect_tx(&b_full[slot], nb * kTcBBox * 128);
          for (int j = 0; j < nb; ++j)
            tma_load_2d(dst + j * kTcBBox * 128, &p.tm_b, s * kTcK, p0 + j * kTcBBox, &b_full[slot]);
        }
      }
      for (int d = gs - kTcSB < 0 ? 0 : gs - kTcSB; d < gs; ++d)
        mbar_wait(&b_full[d % kTcSB], (d / kTcSB) & 1, p.err);
    }
  } else if (warp == kTcWarpMma) {
    if (lane == 0) {
      int gs = 0, lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++lt) {
        const int c = tile / MT;
        const int n16 = (p.w.chunk_n[c] + 15) & ~15;
        const uint32_t idesc = tc::idesc_m128(n16, !F16);
        const int buf = lt & 1;
        if (lt >= 2) ok = tc_wait(&d_empty[buf], ((lt >> 1) - 1) & 1, p.err, dead);
        if (!ok) break;
        tc::fence_after();
        const uint32_t dg = tmem + buf * 128, du = dg + 64;
        for (int s = 0; s < nS; ++s, ++gs) {
          const int as = gs % kTcGuSA, bs = gs % kTcSB;
          ok = tc_wait(&a_full[as], (gs / kTcGuSA) & 1, p.err, dead) &&
               tc_wait(&b_full[bs], (gs / kTcSB) & 1, p.err, dead);
          if (!ok) break;
          tc::fence_after();
          const uint32_t ag = tmem + kTcGuAcol + as * 64, au = ag + 32;
          const uint32_t bsa = smem_addr(bbuf + bs * (kTcCols * 128));
#pragma unroll
          for (int kk = 0; kk < kTcK / 16; ++kk) {
            const uint64_t bd = tc::sdesc_sw128(bsa + 32 * kk);
            const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
            tc::mma_ts(dg, ag + 8 * kk, bd, idesc, acc);
            tc::mma_ts(du, au + 8 * kk, bd, idesc, acc);
          }
          tc::commit(&a_empty[as]);
          tc::commit(&b_empty[bs]);
        }
        if (ok) tc::commit(&d_full[buf]);
      }
      // every MMA done before tensor memory is released
      tc::commit(drain);
      mbar_wait(drain, 0, p.err);
    }
  } else if (warp < kTcWarpEpi + 4) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    int lt = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++lt) {
      const int c = tile / MT, m = tile % MT;
      const int p0 = p.w.chunk_p0[c], n = p.w.chunk_n[c];
      const int buf = lt & 1;
      if (!tc_wait_warp(&d_full[buf], (lt >> 1) & 1, p.err, dead)) break;
      tc::fence_after();
      const int i = m * kTcRows + 32 * q + lane;   // this lane's neuron
      for (int c0 = 0; c0 < n; c0 += 16) {
        uint32_t g[16], u[16];
        tc::ld16(lane_base + buf * 128 + c0, g);
        tc::ld16(lane_base + buf * 128 + 64 + c0, u);
        tc::wait_ld();
        const int myslot = (lane < 16 && c0 + lane < n) ? p.w.pair_slot[p0 + c0 + lane] : 0;
        const float myinv = (F16 && lane < 16 && c0 + lane < n) ? p.w.xinv[p0 + c0 + lane] : 1.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int slot = __shfl_sync(kFull, myslot, j);
          const float inv = F16 ? __shfl_sync(kFull, myinv, j) : 1.f;
          if (c0 + j < n) {
            const float gv = __uint_as_float(g[j]) * inv, uv = __uint_as_float(u[j]) * inv;
            const uint16_t hv = f32_to_bf16_rn((gv / (1.0f + expf(-gv))) * uv);
            p.w.hg[(size_t)(p0 + c0 + j) * I + i] = hv;
            p.h[(size_t)slot * I + i] = hv;
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[buf]);
    }
  } else {
    // --------------------------------------------------------------- decode
    // Warp (quarter q, stage lane j) decodes whole stages for its 32 rows:
    // the stages gs with gs % kTcGuSA == j (so A slot j), gate and up, both
    // 32-element halves; four stages are in decode at once.
    const int dw = warp - kTcFirstDecodeWarp;
    const int q = warp & 3;
    const int j = dw >> 2;
    const int r = 32 * q + lane;                 // row among the tile's gate (and up) rows
    const uint32_t tcol = tmem + ((uint32_t)(32 * q) << 16) + kTcGuAcol + j * 64;
    int gs = 0, gc = 0;
    RingPos rr(R);   // the raw ring's slot and phase (no division by R per stage)
    uint4 scw[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};   // gate, up
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      for (int s = 0; s < nS; ++s, ++gs, rr.next()) {
        if (s % kTcScaleStages == 0) {
          // every decode warp reads every scale chunk (its rows' 16 bytes)
          const int slot = gc % kTcNS;
          ok = tc_wait_warp(&sc_full[slot], (gc / kTcNS) & 1, p.err, dead);
          if (!ok) break;
          const uint8_t* sr = sc + slot * L.scStage + r * 16;
          scw[0] = *reinterpret_cast<const uint4*>(sr);
          scw[1] = *reinterpret_cast<const uint4*>(sr + kTcRows * 16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sc_empty[slot]);
          ++gc;
        }
        if ((gs & (kTcGuSA - 1)) != j) continue;
        ok = tc_wait_warp(&raw_full[rr.slot], rr.phase, p.err, dead);
        if (!ok) break;
        if (gs >= kTcGuSA) ok = tc_wait_warp(&a_empty[j], ((gs / kTcGuSA) - 1) & 1, p.err, dead);
        if (!ok) break;
        tc::fence_after();
        const uint8_t* st = raw + rr.slot * L.rawStage;
#pragma unroll
        for (int b = 0; b < 4; ++b) {   // block b: gate (b < 2) or up, half b & 1
          uint4 cc[2];
          F::load(st + (b >> 1) * kTcRows * RB, r, b & 1, cc);
          const int bi = 2 * (s % kTcScaleStages) + (b & 1);   // block within the scale chunk
          const uint4 w4 = scw[b >> 1];
          const uint32_t word = bi < 4 ? w4.x : bi < 8 ? w4.y : bi < 12 ? w4.z : w4.w;
          uint32_t o[16];
          if constexpr (F16)
            F::decode_f16(cc, (word >> (8 * (bi & 3))) & 0xFFu, o);
          else
            F::decode(cc, (word >> (8 * (bi & 3))) & 0xFFu, o);
          tc::st16(tcol + (b >> 1) * 32 + (b & 1) * 16, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rr.slot]);
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[j]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kTcWarpMma) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, kTcTmemCols);
  }
}

// ---------------------------------------------------------------------------
// moe_tc_down: as moe_tc_gate_up over tiles (chunk c, rows [128 m, 128 m +
// 128) of y), K = I: per stage 128 W_down rows by TMA, their scales once a
// tile (a bulk copy of 128 rows of I/32 bytes), 8 decode warps (quarter x
// every other stage), the chunk's hg rows as B, 4 MMAs into one accumulator; the epilogue
// writes the pairs' FP32 partial rows yp[p][128 m ...].
// ---------------------------------------------------------------------------
template <class F>
__global__ void __launch_bounds__(kTcDnThreads, 1) moe_tc_down(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int RB = F::kStageRowBytes;
  const int R = p.R;
  const TcSmem L(true, RB, R, p.I);
  uint8_t* raw = smem + L.raw;
  uint8_t* bbuf = smem + L.b;
  uint8_t* sc = smem + L.sc;
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* raw_empty = raw_full + R;
  uint64_t* b_full = raw_empty + R;
  uint64_t* b_empty = b_full + kTcSB;
  uint64_t* a_full = b_empty + kTcSB;
  uint64_t* a_empty = a_full + kTcDnSA;
  uint64_t* sc_full = a_empty + kTcDnSA;
  uint64_t* sc_empty = sc_full + 2;
  uint64_t* d_full = sc_empty + 2;
  uint64_t* d_empty = d_full + 2;
  uint64_t* drain = d_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* dead = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, I = p.I, nbI = I / 32;
  const int nS = I / kTcK;          // stages a tile
  const int MT = H / kTcRows;       // row tiles an expert

  if (warp == kTcWarpRaw && lane == 0) tc::prefetch_tmap(&p.tm_w);
  if (warp == kTcWarpB && lane == 0) tc::prefetch_tmap(&p.tm_b);
  if (warp == kTcWarpEpi && lane == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], 4);   // the four lane quarters' decode warps of the stage
    }
    for (int i = 0; i < kTcSB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kTcDnSA; ++i) {
      mbar_init(&a_full[i], 4);      // the four lane quarters' decode warps of the stage
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sc_full[i], 1);
      mbar_init(&sc_empty[i], kTcDnDecodeWarps);
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 4);
    }
    mbar_init(drain, 1);
    *dead = 0;
    mbar_init_fence();
  }
  if (warp == kTcWarpMma) tc::tmem_alloc(tmem_slot, kTcTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // hg comes from moe_tc_gate_up
  const int ntiles = p.w.hdr[2] * MT;

  if (warp == kTcWarpRaw) {
    if (lane == 0) {
      int gs = 0, lt = 0;
      RingPos rw(R);   // the raw ring's slot and phase (no division by R per stage)
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++lt) {
        const int c = tile / MT, m = tile % MT;
        const size_t row0 = (size_t)p.w.chunk_e[c] * H + (size_t)m * kTcRows;
        const int ss = lt & 1;
        if (lt >= 2) ok = tc_wait(&sc_empty[ss], ((lt >> 1) - 1) & 1, p.err, dead);
        if (!ok) break;
        mbar_expect_tx(&sc_full[ss], kTcRows * nbI);
        bulk_copy_g2s(sc + ss * L.scStage, p.sd + row0 * nbI, kTcRows * nbI, &sc_full[ss]);
        for (int s = 0; s < nS; ++s, ++gs) {
          const int slot = rw.slot;
          if (gs >= R) ok = tc_wait(&raw_empty[slot], rw.phase ^ 1u, p.err, dead);
          if (!ok) break;
          mbar_expect_tx(&raw_full[slot], L.rawStage);
          tma_load_2d(raw + slot * L.rawStage, &p.tm_w, s * RB, (int)row0, &raw_full[slot]);
          rw.next();
        }
      }
      for (int d = gs - R < 0 ? 0 : gs - R; d < gs; ++d) mbar_wait(&raw_full[d % R], (d / R) & 1, p.err);
      for (int d = lt - 2 < 0 ? 0 : lt - 2; d < lt; ++d) mbar_wait(&sc_full[d & 1], (d >> 1) & 1, p.err);
    }
  } else if (warp == kTcWarpB) {
    if (lane == 0) {
      int gs = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
        const int c = tile / MT;
        const int p0 = p.w.chunk_p0[c], nb = (p.w.chunk_n[c] + kTcBBox - 1) / kTcBBox;
        for (int s = 0; s < nS; ++s, ++gs) {
          const int slot = gs % kTcSB;
          if (gs >= kTcSB) ok = tc_wait(&b_empty[slot], ((gs / kTcSB) - 1) & 1, p.err, dead);
          if (!ok) break;
          uint8_t* dst = bbuf + slot * (kTcCols * 128);
          mbar_expect_tx(&b_full[slot], nb * kTcBBox * 128);
          for (int j = 0; j < nb; ++j)
            tma_load_2d(dst + j * kTcBBox * 128, &p.tm_b, s * kTcK, p0 + j * kTcBBox, &b_full[slot]);
        }
      }
      for (int d = gs - kTcSB < 0 ? 0 : gs - kTcSB; d < gs; ++d)
        mbar_wait(&b_full[d % kTcSB], (d / kTcSB) & 1, p.err);
    }
  } else if (warp == kTcWarpMma) {
    if (lane == 0) {
      int gs = 0, lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++lt) {
        const int c = tile / MT;
        const uint32_t idesc = tc::idesc_m128((p.w.chunk_n[c] + 15) & ~15, true);
        const int buf = lt & 1;
        if (lt >= 2) ok = tc_wait(&d_empty[buf], ((lt >> 1) - 1) & 1, p.err, dead);
        if (!ok) break;
        tc::fence_after();
        const uint32_t dd = tmem + buf * kTcCols;
        for (int s = 0; s < nS; ++s, ++gs) {
          const int as = gs % kTcDnSA, bs = gs % kTcSB;
          ok = tc_wait(&a_full[as], (gs / kTcDnSA) & 1, p.err, dead) &&
               tc_wait(&b_full[bs], (gs / kTcSB) & 1, p.err, dead);
          if (!ok) break;
          tc::fence_after();
          const uint32_t a = tmem + kTcDnAcol + as * 32;
          const uint32_t bsa = smem_addr(bbuf + bs * (kTcCols * 128));
#pragma unroll
          for (int kk = 0; kk < kTcK / 16; ++kk)
            tc::mma_ts(dd, a + 8 * kk, tc::sdesc_sw128(bsa + 32 * kk), idesc,
                       (s > 0 || kk > 0) ? 1u : 0u);
          tc::commit(&a_empty[as]);
          tc::commit(&b_empty[bs]);
        }
        if (ok) tc::commit(&d_full[buf]);
      }
      tc::commit(drain);
      mbar_wait(drain, 0, p.err);
    }
  } else if (warp < kTcWarpEpi + 4) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    int lt = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++lt) {
      const int c = tile / MT, m = tile % MT;
      const int p0 = p.w.chunk_p0[c], n = p.w.chunk_n[c];
      const int buf = lt & 1;
      if (!tc_wait_warp(&d_full[buf], (lt >> 1) & 1, p.err, dead)) break;
      tc::fence_after();
      float* out = p.w.yp + (size_t)p0 * H + m * kTcRows + 32 * q + lane;
      for (int c0 = 0; c0 < n; c0 += 16) {
        uint32_t v[16];
        tc::ld16(lane_base + buf * kTcCols + c0, v);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < n) out[(size_t)(c0 + j) * H] = __uint_as_float(v[j]);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[buf]);
    }
  } else {
    // --------------------------------------------------------------- decode
    // Warp (quarter q, stage lane j) decodes whole stages for its 32 rows:
    // the stages gs with gs % kTcDnLanes == j, both 32-element halves.
    const int dw = warp - kTcFirstDecodeWarp;
    const int q = warp & 3, j = dw >> 2;
    const int r = 32 * q + lane;
    const uint32_t tcol = tmem + ((uint32_t)(32 * q) << 16) + kTcDnAcol;
    int gs = 0, lt = 0;
    RingPos rr(R);   // the raw ring's slot and phase (no division by R per stage)
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++lt) {
      const int ss = lt & 1;
      ok = tc_wait_warp(&sc_full[ss], (lt >> 1) & 1, p.err, dead);
      if (!ok) break;
      const uint8_t* srow = sc + ss * L.scStage + r * nbI;
      for (int s = 0; s < nS; ++s, ++gs, rr.next()) {
        if ((gs & (kTcDnLanes - 1)) != j) continue;
        const int slot = rr.slot;
        ok = tc_wait_warp(&raw_full[slot], rr.phase, p.err, dead);
        if (!ok) break;
        const int as = gs % kTcDnSA;
        if (gs >= kTcDnSA) ok = tc_wait_warp(&a_empty[as], ((gs / kTcDnSA) - 1) & 1, p.err, dead);
        if (!ok) break;
        tc::fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint4 cc[2];
          F::load(raw + slot * L.rawStage, r, half, cc);
          uint32_t o[16];
          F::decode(cc, srow[2 * s + half], o);
          tc::st16(tcol + as * 32 + half * 16, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[slot]);
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc_empty[ss]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kTcWarpMma) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, kTcTmemCols);
  }
}

// ---------------------------------------------------------------------------
// moe_tc_combine: y[t, r] = bf16(sum_j topk_w[t, j] * yp[pair(t, j), r]) over
// the slots with valid ids, in slot order (the warp-decode post, "How the two
// kernels work": the routing-weighted sum over the top-k experts). Grid
// (H / 1024 rounded up, T); four rows a thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTcCombineThreads) moe_tc_combine(const __grid_constant__ TcCombineParams p) {
  pdl_wait();   // yp comes from moe_tc_down
  pdl_trigger();
  const int t = blockIdx.y;
  const int r = (blockIdx.x * kTcCombineThreads + threadIdx.x) * 4;
  if (r >= p.H) return;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  for (int j = 0; j < p.k; ++j) {
    const int q = p.w.slot_pair[t * p.k + j];
    if (q < 0) continue;
    const float wj = __ldg(p.tw + t * p.k + j);
    const float4 v = *reinterpret_cast<const float4*>(p.w.yp + (size_t)q * p.H + r);
    a0 = fmaf(wj, v.x, a0);
    a1 = fmaf(wj, v.y, a1);
    a2 = fmaf(wj, v.z, a2);
    a3 = fmaf(wj, v.w, a3);
  }
  uint16_t* y = p.y + (size_t)t * p.H + r;
  y[0] = f32_to_bf16_rn(a0);
  y[1] = f32_to_bf16_rn(a1);
  y[2] = f32_to_bf16_rn(a2);
  y[3] = f32_to_bf16_rn(a3);
}

// ---------------------------------------------------------------------------
// moe_tc_scan: whether every weight decodes exactly to a normal bf16 -- out[0]
// the smallest scale code, out[1] the largest, out[2] set when an E4M3 code
// is NaN (byte & 0x7F == 0x7F). Both arrays as 16-byte words.
// ---------------------------------------------------------------------------
__global__ void moe_tc_scan(const uint4* codes, size_t ncodes16, const uint4* scales,
                            size_t nscales16, int fp8, uint32_t* out) {
  uint32_t lo = 0xFFFFFFFFu, hi = 0u, nan = 0u;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nscales16; i += stride) {
    const uint4 v = scales[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t s = (w[j] >> (8 * b)) & 0xFFu;
        lo = min(lo, s);
        hi = max(hi, s);
      }
    }
  }
  if (fp8) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < ncodes16; i += stride) {
      const uint4 v = codes[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) nan |= ((w[j] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(kFull, lo, o));
    hi = max(hi, __shfl_xor_sync(kFull, hi, o));
    nan |= __shfl_xor_sync(kFull, nan, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&out[0], lo);
    atomicMax(&out[1], hi);
    if (nan) atomicOr(&out[2], 1u);
  }
}

}  // namespace moe
