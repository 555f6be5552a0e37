// The whole single-token layer in one persistent launch.
//
// Both projections of the warp-decode post (cursor.com/blog/warp-decode, "How
// the two kernels work") run here as two phases of one cooperative kernel with
// one CTA per SM. The split of work is the post's output-centric one: in the
// gate/up phase a warp owns one intermediate neuron and reduces its gate and
// up dot products itself; in the down phase a warp owns one output row.
//
// What the single launch adds is the memory stream. One producer warp per CTA
// feeds two rings of shared-memory slots guarded by mbarriers: the gate/up
// ring (TMA tensor tiles of fifteen neurons' gate and up rows over a K-chunk)
// and the down ring (bulk copies of the CTA's output rows of one routed
// expert). Gate/up tiles go first; whenever the gate/up ring is full the
// producer fills free down slots instead, so HBM keeps streaming while the
// consumers compute, and by the time the fifteen consumer warps have written
// h and passed the grid barrier most of their down rows are already on chip.
//
// Arithmetic. Each lane reduces one 32-element MX block at a time: 32 E4M3
// codes against 32 activations, FP32 accumulation, then the block's UE8M0
// scale. The activations (x in the gate/up phase, h in the down phase) are
// held in shared memory as f16 after multiplying each 32-element block by a
// power of two 2^e that brings its largest magnitude into [2^14, 2^15); the
// factor 2^-e is applied to the block's sum. E4M3 -> f16 is exact, a bf16
// value scaled that way is exact in f16 whenever it lies within 2^-28 of its
// block's largest magnitude, and an f16 x f16 product is exact in FP32, so
// fma.rn.f32.f16 gives the same sums as FP32 FMAs on the decoded values.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "moe_kernels.cuh"

namespace moe {

// 15 consumer warps + 1 producer warp: 4 warps per SM sub-partition, so each
// thread may hold up to 128 registers (a sub-partition has 16K).
constexpr int kFusedConsumers = 15;                       // consumer warps
constexpr int kFusedThreads = (kFusedConsumers + 1) * 32; // + one producer warp
constexpr int kFusedNeurons = kFusedConsumers;            // gate/up neurons per stage

struct FusedParams {
  // W_gateup codes and scales as 2D uint32 tensors ([E*2I, H/4] and
  // [E*2I, H/128]), boxes of kFusedNeurons rows x KC codes (x KC/32 scale bytes)
  CUtensorMap tm_codes;
  CUtensorMap tm_scales;
  const uint16_t* x;          // [1, H] bf16
  const int32_t* ids;         // [1, k]
  const float* w;             // [1, k]
  const uint8_t* wgu;         // [E, 2I, H]
  const uint8_t* sgu;         // [E, 2I, H/32]
  const uint8_t* wd;          // [E, H, I]
  const uint8_t* sd;          // [E, H, I/32]
  uint16_t* h;                // [1, k, I] bf16 (written, then read back through L2)
  uint16_t* y;                // [1, H] bf16
  uint32_t* err;
  unsigned long long* grid_bar;   // arrivals, grows by gridDim.x per launch
  int k, E, H, I;
  int KC;       // gate/up codes per row per stage: 512 or 1024, divides H
  int SG;       // gate/up ring slots
  int slot_g;   // bytes per gate/up slot (GuStageLayout(KC).end)
  int SD;       // down slots (one routed expert's row chunk each), filled as one group
  int slot_d;   // bytes per down slot: RC rows of codes, then RC rows of scales
  int RG;       // down row granule (keeps scale copies 16-byte aligned)
  int RC;       // down rows per chunk (multiple of RG, <= kFusedConsumers)
};

__host__ __device__ constexpr int round128(int v) { return (v + 127) / 128 * 128; }

// Byte offsets of a gate/up stage in a ring slot: gate codes, up codes, gate
// scales, up scales, each region starting on a 128-byte boundary (the TMA
// tensor copies that fill them require it); `end` is the bytes used.
struct GuStageLayout {
  int up, gs, us, end;
  __host__ __device__ explicit GuStageLayout(int KC)
      : up(round128(kFusedNeurons * KC)),
        gs(2 * round128(kFusedNeurons * KC)),
        us(2 * round128(kFusedNeurons * KC) + round128(kFusedNeurons * (KC >> 5))),
        end(2 * round128(kFusedNeurons * KC) + 2 * round128(kFusedNeurons * (KC >> 5))) {}
};

// Shared-memory map of the kernel (byte offsets, each 128-byte aligned).
struct FusedSmem {
  int ring_d;   // SD down slots (the SG gate/up slots start at 0)
  int xs;       // x as f16, [H/32] blocks of 64 bytes (swizzled 16-byte chunks)
  int xf;       // [H/32] FP32 block factors 2^-e of x
  int hs;       // h of each unique expert as f16, [k][I/32] blocks of 64 bytes
  int hf;       // [k][I/32] FP32 block factors of h
  int cf;       // [k] combined routing weight of each unique expert
  int jz;       // [k] first slot j routed to each unique expert
  int bars;     // mbarriers: full_g[SG], empty_g[SG], full_d, empty_d
  int words;    // 16 warps x 32 words of expert bitmap
  int total;
  __host__ __device__ FusedSmem(int SG, int slot_g, int SD, int slot_d, int H, int I, int k) {
    int o = SG * slot_g;
    ring_d = o;
    o += SD * slot_d;
    xs = o;
    o += round128(H * 2);
    xf = o;
    o += round128((H >> 5) * 4);
    hs = o;
    o += round128(k * I * 2);
    hf = o;
    o += round128(k * (I >> 5) * 4);
    cf = o;
    o += round128(k * 4);
    jz = o;
    o += round128(k * 4);
    bars = o;
    o += round128((2 * SG + 2) * 8);
    words = o;
    o += 16 * 32 * 4;
    total = o;
  }
};

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

// The CTA's gate/up stage sequence: up to 15 neurons of one expert over a
// K-chunk (u-major over the unique experts). Producer and consumers run the
// same warp-uniform walk; it steps without divisions.
struct GuWalk {
  int g, g1;          // neuron cursor and end of the CTA's slice
  int u, i0, nn, kc, nkc, I;
  bool valid;

  __device__ __forceinline__ void set_nn() {
    valid = g < g1;
    nn = kFusedNeurons;
    if (nn > I - i0) nn = I - i0;
    if (nn > g1 - g) nn = g1 - g;
  }
  __device__ __forceinline__ void begin(int nU, const FusedParams& p) {
    I = p.I;
    nkc = p.H / p.KC;
    const long long G = (long long)nU * I;
    g = (int)(G * blockIdx.x / gridDim.x);
    g1 = (int)(G * (blockIdx.x + 1) / gridDim.x);
    u = g / I;
    i0 = g - u * I;
    kc = 0;
    set_nn();
  }
  __device__ __forceinline__ void next() {
    if (++kc < nkc) return;
    kc = 0;
    g += nn;
    i0 += nn;
    if (i0 == I) {
      i0 = 0;
      ++u;
    }
    set_nn();
  }
  __device__ __forceinline__ bool last_kc() const { return kc == nkc - 1; }
};

// The CTA's down work: output rows [r0, r1) (whole granules of RG rows), cut
// in chunks of RC rows; each chunk's unique experts in groups of up to SD
// (one expert per down slot). A group is loaded and consumed as one unit.
struct DownWalk {
  int r0, r1, c0, rc, u0, ng, nU, RC, SD;
  bool valid;

  __device__ __forceinline__ void begin(int nU_, const FusedParams& p) {
    const int nrg = p.H / p.RG;
    r0 = (int)((long long)nrg * blockIdx.x / gridDim.x) * p.RG;
    r1 = (int)((long long)nrg * (blockIdx.x + 1) / gridDim.x) * p.RG;
    nU = nU_;
    RC = p.RC;
    SD = p.SD;
    c0 = r0;
    u0 = 0;
    valid = r0 < r1 && nU > 0;
    rc = (r1 - c0) < RC ? (r1 - c0) : RC;
    ng = nU < SD ? nU : SD;
  }
  __device__ __forceinline__ void next() {
    u0 += ng;
    if (u0 >= nU) {
      u0 = 0;
      c0 += rc;
      valid = c0 < r1;
      rc = (r1 - c0) < RC ? (r1 - c0) : RC;
    }
    ng = (nU - u0) < SD ? (nU - u0) : SD;
  }
  __device__ __forceinline__ bool last_group() const { return u0 + ng >= nU; }
};

// Ring position: slot index and the parity of its current fill.
struct RingPos {
  int slot, n;
  uint32_t phase;
  __device__ __forceinline__ RingPos(int n_) : slot(0), n(n_), phase(0) {}
  __device__ __forceinline__ void next() {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Grid-wide barrier for a cooperative launch: every CTA adds one arrival to a
// 64-bit counter that grows by gridDim.x per launch (a release at GPU scope,
// after the CTA's threads met at a named barrier), then polls it with acquire
// loads (bounded) until this launch's arrivals are complete. Called by one
// thread per CTA.
__device__ __forceinline__ bool grid_barrier(unsigned long long* bar, uint32_t* err) {
  unsigned long long ticket;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;" : "=l"(ticket) : "l"(bar) : "memory");
  const unsigned long long G = gridDim.x;
  const unsigned long long target = (ticket / G + 1) * G;
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(bar) : "memory");
    if (v >= target) return true;
  }
  atomicOr(err, kDeviceTimeout);
  return false;
}

template <int KMAX>
__global__ void __launch_bounds__(kFusedThreads, 1) moe_layer_fused_t1(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = p.H, I = p.I, KC = p.KC, SG = p.SG, nbI = I >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const FusedSmem L(SG, p.slot_g, p.SD, p.slot_d, H, I, p.k);
  uint8_t* ring_g = smem;
  uint8_t* ring_d = smem + L.ring_d;
  uint8_t* xs = smem + L.xs;
  float* xf = reinterpret_cast<float*>(smem + L.xf);
  uint8_t* hs = smem + L.hs;
  float* hf = reinterpret_cast<float*>(smem + L.hf);
  float* cf = reinterpret_cast<float*>(smem + L.cf);
  int* jz = reinterpret_cast<int*>(smem + L.jz);
  uint64_t* full_g = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty_g = full_g + SG;
  uint64_t* full_d = empty_g + SG;    // one barrier pair for the down group buffer
  uint64_t* empty_d = full_d + 1;
  uint32_t* sm_words = reinterpret_cast<uint32_t*>(smem + L.words);
  const int ctid = threadIdx.x;                    // consumer thread index
  const int ncons = kFusedConsumers * 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < SG; ++i) {
      mbar_init(&full_g[i], 1);
      mbar_init(&empty_g[i], kFusedConsumers);
    }
    mbar_init(full_d, 1);
    mbar_init(empty_d, kFusedConsumers);
    mbar_init_fence();
  }
  __syncthreads();
  pdl_wait();      // x, topk_ids and topk_w come from upstream work
  pdl_trigger();
  if (warp < kFusedConsumers) {
    // x -> f16 blocks first: these loads go out before the weight stream
    for (int b = ctid; b < (H >> 5); b += ncons) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x) + 4 * b;
      const uint4 v[4] = {__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3)};
      xf[b] = stage_block_f16(v, xs + 64 * b, b);
    }
  }
  WarpSchedule<KMAX> s;
  s.build(p.ids, 1, p.k, p.E, sm_words + warp * 32, p.err);
  const int nU = s.n_unique;
  const GuStageLayout lay(KC);

  if (warp == kFusedConsumers) {
    // ------------------------------------------------------------ producer
    GuWalk gw;
    gw.begin(nU, p);
    DownWalk dw;
    dw.begin(nU, p);
    RingPos rg(SG);
    uint32_t dphase = 0;
    int gi = 0, dgroups = 0;
    bool ok = true;
    while (gw.valid || dw.valid) {
      // 1: a gate/up stage, 2: a down group
      int what = 0;
      if (gw.valid) {
        bool free_slot = gi < SG;
        if (!free_slot && lane == 0) free_slot = mbar_test(&empty_g[rg.slot], rg.phase ^ 1u);
        if (__shfl_sync(kFull, free_slot, 0)) what = 1;
      }
      // the first down group's buffer is free from the start; later groups are
      // only waited for once no gate/up stage is left (their consumers come after)
      if (!what && dw.valid && (dgroups == 0 || !gw.valid)) what = 2;
      if (!what) {
        if (lane == 0) ok = mbar_wait(&empty_g[rg.slot], rg.phase ^ 1u, p.err);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
        what = 1;
      }
      if (what == 1) {
        const int e = s.expert(gw.u);   // warp-collective
        if (lane == 0) {
          uint8_t* dst = ring_g + (size_t)rg.slot * p.slot_g;
          uint64_t* bar = &full_g[rg.slot];
          // four tensor copies: the stage's gate rows, up rows, and their scales
          // (full boxes; rows past the expert are never read)
          mbar_expect_tx(bar, 2u * kFusedNeurons * KC + 2u * kFusedNeurons * (KC >> 5));
          const int row = e * 2 * I + gw.i0;
          tma_load_2d(dst, &p.tm_codes, gw.kc * (KC >> 2), row, bar);
          tma_load_2d(dst + lay.up, &p.tm_codes, gw.kc * (KC >> 2), row + I, bar);
          tma_load_2d(dst + lay.gs, &p.tm_scales, gw.kc * (KC >> 7), row, bar);
          tma_load_2d(dst + lay.us, &p.tm_scales, gw.kc * (KC >> 7), row + I, bar);
        }
        gw.next();
        rg.next();
        ++gi;
      } else {
        if (lane == 0 && dgroups > 0) ok = mbar_wait(empty_d, dphase ^ 1u, p.err);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
        const uint32_t cb = (uint32_t)dw.rc * I, sb = (uint32_t)dw.rc * nbI;
        if (lane == 0) mbar_expect_tx(full_d, (cb + sb) * dw.ng);
        for (int gi2 = 0; gi2 < dw.ng; ++gi2) {
          const int e = s.expert(dw.u0 + gi2);   // warp-collective
          if (lane == 0) {
            uint8_t* dst = ring_d + (size_t)gi2 * p.slot_d;
            const size_t row = (size_t)e * H + dw.c0;
            bulk_copy_g2s(dst, p.wd + row * I, cb, full_d);
            bulk_copy_g2s(dst + (size_t)p.RC * I, p.sd + row * nbI, sb, full_d);
          }
        }
        dw.next();
        dphase ^= 1u;
        ++dgroups;
      }
    }
    // never leave with copies in flight: the last stages of each ring must land
    if (lane == 0) {
      RingPos r(SG);
      for (int d = 0; d < gi; ++d, r.next())
        if (d >= gi - SG) mbar_wait(&full_g[r.slot], r.phase, p.err);
      if (dgroups > 0) mbar_wait(full_d, dphase ^ 1u, p.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  named_sync(1, ncons);   // x staged
  // per unique expert: the combined routing weight of its slots and the first
  // slot routed to it (its h row); out-of-range ids give h = 0 (written by
  // CTA 0) and no down term
  if (warp == 0) {
    const float wj = (lane < p.k) ? __ldg(p.w + lane) : 0.f;
    for (int u = 0; u < nU; ++u) {
      const int e = s.expert(u);
      const uint32_t jm = __shfl_sync(kFull, s.jmask(e), 0);   // lane 0 holds the token
      const float c = warp_sum(((jm >> lane) & 1u) ? wj : 0.f);
      if (lane == 0) {
        cf[u] = c;
        jz[u] = __ffs(jm) - 1;
      }
    }
    if (blockIdx.x == 0 && s.badmask) {
      for (uint32_t m = s.badmask; m; m &= m - 1) {
        uint16_t* row = p.h + (size_t)(__ffs(m) - 1) * I;
        for (int i = 0; i < I; ++i) row[i] = 0;   // lane 0 alone holds the token
      }
    }
  }

  const LaneBlock lb(lane);
  // a warp whose bounded wait gave up stops waiting and computing but still
  // reaches every arrival and named barrier, so no other warp can hang on it
  bool dead = false;

  // ---- gate/up: warp owns neuron i0 + warp of each stage, lane owns block lane
  {
    GuWalk gw;
    gw.begin(nU, p);
    RingPos rg(SG);
    float ag = 0.f, au = 0.f;
    const int nbk = KC >> 5;                      // blocks per row per stage
    for (; gw.valid; gw.next(), rg.next()) {
      if (!dead) dead = !mbar_wait(&full_g[rg.slot], rg.phase, p.err);
      if (warp < gw.nn && !dead) {
        const uint8_t* base = ring_g + (size_t)rg.slot * p.slot_g;
        for (int bl = lane; bl < nbk; bl += 32) {
          const int b = gw.kc * nbk + bl;         // block of the H row
          const uint8_t* act = xs + 64 * b;
          const float fx = xf[b];
          const float dg = dot_block(base + warp * KC + 32 * bl, act, lb);
          const float du = dot_block(base + lay.up + warp * KC + 32 * bl, act, lb);
          ag = fmaf(dg * fx, ue8m0_to_f32(base[lay.gs + warp * nbk + bl]), ag);
          au = fmaf(du * fx, ue8m0_to_f32(base[lay.us + warp * nbk + bl]), au);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_g[rg.slot]);
      if (gw.last_kc()) {
        const int e = s.expert(gw.u);   // warp-collective
        if (warp < gw.nn) {
          const float g = warp_sum(ag);
          const float up = warp_sum(au);
          const uint32_t jm = __shfl_sync(kFull, s.jmask(e), 0);
          const uint16_t hb = f32_to_bf16_rn((g / (1.0f + expf(-g))) * up);
          if (lane < p.k && ((jm >> lane) & 1u)) p.h[(size_t)lane * I + gw.i0 + warp] = hb;
        }
        ag = au = 0.f;
      }
    }
  }

  // every h value of every CTA is written before any CTA reads h
  named_sync(1, ncons);
  if (ctid == 0 && !grid_barrier(p.grid_bar, p.err)) dead = true;
  named_sync(1, ncons);
  // h of each unique expert -> f16 blocks (read through L2: other CTAs wrote it)
  for (int t = ctid; t < nU * nbI; t += ncons) {
    const int u = t / nbI, b = t - u * nbI;
    const uint4* src = reinterpret_cast<const uint4*>(p.h + (size_t)jz[u] * I) + 4 * b;
    const uint4 v[4] = {__ldcg(src), __ldcg(src + 1), __ldcg(src + 2), __ldcg(src + 3)};
    hf[t] = stage_block_f16(v, hs + 64 * t, b);
  }
  named_sync(1, ncons);

  // ---- down: warp owns row c0 + warp of each chunk; its lanes take the
  // group's (expert, block) pairs, two at a time
  {
    DownWalk dw;
    dw.begin(nU, p);
    uint32_t dphase = 0;
    float acc = 0.f;
    for (; dw.valid; dw.next(), dphase ^= 1u) {
      if (!dead) dead = !mbar_wait(full_d, dphase, p.err);
      if (warp < dw.rc && !dead) {
        const int n_items = dw.ng * nbI;
        // item t: expert ui = t / nbI of the group, block b = t % nbI
        int ui = 0, b = lane;
        while (b >= nbI) { b -= nbI; ++ui; }
        for (int t = lane; t < n_items; t += 64) {
          // this item and the one 32 further on
          int ui2 = ui, b2 = b + 32;
          while (b2 >= nbI) { b2 -= nbI; ++ui2; }
          const bool two = t + 32 < n_items;
          const uint8_t* s1 = ring_d + (size_t)ui * p.slot_d;
          const float d1 = dot_block(s1 + (size_t)warp * I + 32 * b, hs + (size_t)(dw.u0 + ui) * nbI * 64 + 64 * b, lb);
          float d2 = 0.f;
          const uint8_t* s2 = ring_d + (size_t)ui2 * p.slot_d;
          if (two) d2 = dot_block(s2 + (size_t)warp * I + 32 * b2, hs + (size_t)(dw.u0 + ui2) * nbI * 64 + 64 * b2, lb);
          const float v1 = d1 * hf[(dw.u0 + ui) * nbI + b] * ue8m0_to_f32(s1[(size_t)p.RC * I + warp * nbI + b]);
          acc = fmaf(v1, cf[dw.u0 + ui], acc);
          if (two) {
            const float v2 = d2 * hf[(dw.u0 + ui2) * nbI + b2] * ue8m0_to_f32(s2[(size_t)p.RC * I + warp * nbI + b2]);
            acc = fmaf(v2, cf[dw.u0 + ui2], acc);
          }
          // advance both cursors by 64 items
          ui = ui2;
          b = b2 + 32;
          while (b >= nbI) { b -= nbI; ++ui; }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_d);
      if (dw.last_group()) {
        const float v = warp_sum(acc);
        if (lane == 0 && warp < dw.rc) p.y[dw.c0 + warp] = f32_to_bf16_rn(v);
        acc = 0.f;
      }
    }
    if (nU == 0) {
      // no valid expert at all: the CTA's output rows are zero
      for (int r = dw.r0 + ctid; r < dw.r1; r += ncons) p.y[r] = 0;
    }
  }
}

}  // namespace moe
