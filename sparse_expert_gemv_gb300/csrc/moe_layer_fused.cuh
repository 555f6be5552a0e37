// The whole single-token layer in one persistent launch.
//
// Both projections of the warp-decode post (cursor.com/blog/warp-decode, "How
// the two kernels work") run here as two phases of one cooperative kernel with
// one CTA per SM. The split of work is the posts' output-centric one: in the
// gate/up phase a warp owns one intermediate neuron and reduces its gate and
// up dot products itself; in the down phase a warp owns one output row.
//
// What the single launch adds is the memory stream. One producer warp per CTA
// issues cp.async.bulk copies of the CTA's gate/up row blocks and, right after
// them, of the CTA's down rows for every routed expert, into one ring of
// shared-memory slots guarded by mbarriers. HBM therefore never waits for the
// gate/up arithmetic to finish before the down weights are requested: by the
// time the fifteen consumer warps have written h and passed the grid barrier,
// their down rows are already in shared memory.
#pragma once

#include <cuda.h>

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
  int KC;           // gate/up codes per row per stage: 512 or 1024, divides H
  int S;            // ring slots
  int slot_bytes;   // bytes per slot (multiple of 128)
  int RG;           // down row granule (keeps scale copies 16-byte aligned)
  int RC;           // down rows per stage (multiple of RG, <= kFusedConsumers)
  int GE;           // experts per down stage
  int EB;           // bytes per expert inside a down stage (multiple of 16)
};

// Byte offsets of a gate/up stage in a ring slot: gate codes, up codes, gate
// scales, up scales, each region starting on a 128-byte boundary (the TMA
// tensor copies that fill them require it); `end` is the bytes used.
struct GuStageLayout {
  int up, gs, us, end;
  __host__ __device__ static constexpr int r128(int v) { return (v + 127) / 128 * 128; }
  __host__ __device__ explicit GuStageLayout(int KC)
      : up(r128(kFusedNeurons * KC)),
        gs(2 * r128(kFusedNeurons * KC)),
        us(2 * r128(kFusedNeurons * KC) + r128(kFusedNeurons * (KC >> 5))),
        end(2 * r128(kFusedNeurons * KC) + 2 * r128(kFusedNeurons * (KC >> 5))) {}
};

// float4 slot of quarter jj of piece q (16 FP32 values): an XOR swizzle so that
// eight lanes reading eight consecutive pieces hit eight distinct bank groups.
__device__ __forceinline__ int piece_slot(int q, int jj) { return q * 4 + (jj ^ ((q >> 1) & 3)); }

// 16 E4M3 codes (one uint4) dotted with 16 FP32 values (four float4).
__device__ __forceinline__ float dot16(const uint4 q, const float4 x0, const float4 x1,
                                       const float4 x2, const float4 x3) {
  float w[16];
  e4m3x4_to_f32(q.x, w[0], w[1], w[2], w[3]);
  e4m3x4_to_f32(q.y, w[4], w[5], w[6], w[7]);
  e4m3x4_to_f32(q.z, w[8], w[9], w[10], w[11]);
  e4m3x4_to_f32(q.w, w[12], w[13], w[14], w[15]);
  float a = w[0] * x0.x;
  float b = w[1] * x0.y;
  a = fmaf(w[2], x0.z, a);
  b = fmaf(w[3], x0.w, b);
  a = fmaf(w[4], x1.x, a);
  b = fmaf(w[5], x1.y, b);
  a = fmaf(w[6], x1.z, a);
  b = fmaf(w[7], x1.w, b);
  a = fmaf(w[8], x2.x, a);
  b = fmaf(w[9], x2.y, b);
  a = fmaf(w[10], x2.z, a);
  b = fmaf(w[11], x2.w, b);
  a = fmaf(w[12], x3.x, a);
  b = fmaf(w[13], x3.y, b);
  a = fmaf(w[14], x3.z, a);
  b = fmaf(w[15], x3.w, b);
  return a + b;
}

// bf16 vector [n] (n % 16 == 0) -> swizzled FP32 pieces; `nthr` threads share it.
// Reads go through L2 only (ld.global.cg): the data may have been written by
// other CTAs of this launch.
__device__ __forceinline__ void stage_f32_pieces(const uint16_t* __restrict__ src, int n,
                                                 float4* __restrict__ dst, int tid, int nthr) {
  for (int c = tid; c < (n >> 3); c += nthr) {
    const uint4 v = __ldcg(reinterpret_cast<const uint4*>(src) + c);
    const int q = c >> 1, jj = (c & 1) * 2;
    dst[piece_slot(q, jj)] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    dst[piece_slot(q, jj + 1)] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
  }
}

// The CTA's stage sequence: gate/up stages (15 neurons of one expert over a
// K-chunk), then down stages (a chunk of the CTA's rows for up to GE unique
// experts). Producer and consumers run the same warp-uniform walk.
struct FusedWalk {
  // gate/up part
  long long g, g1;    // neuron cursor and end of the CTA's slice (u-major)
  int u, i0, nn, kc, nkc;
  // down part
  int r0, r1, c0, rc, u0, ng;
  int I, nU, RC, GE;
  bool down, valid;

  __device__ __forceinline__ void open_gu() {
    valid = g < g1;
    if (!valid) return;
    u = (int)(g / I);
    i0 = (int)(g - (long long)u * I);
    nn = kFusedNeurons;
    if (nn > I - i0) nn = I - i0;
    if (nn > g1 - g) nn = (int)(g1 - g);
    kc = 0;
  }

  __device__ __forceinline__ void open_down() {
    down = true;
    c0 = r0;
    u0 = 0;
    valid = r0 < r1 && nU > 0;
    if (valid) {
      rc = (r1 - c0) < RC ? (r1 - c0) : RC;
      ng = (nU - u0) < GE ? (nU - u0) : GE;
    }
  }

  __device__ __forceinline__ void begin(int nU_, const FusedParams& p) {
    I = p.I;
    nU = nU_;
    RC = p.RC;
    GE = p.GE;
    nkc = p.H / p.KC;
    const long long G = (long long)nU * I;
    g = G * blockIdx.x / gridDim.x;
    g1 = G * (blockIdx.x + 1) / gridDim.x;
    const int nrg = p.H / p.RG;
    r0 = (int)((long long)nrg * blockIdx.x / gridDim.x) * p.RG;
    r1 = (int)((long long)nrg * (blockIdx.x + 1) / gridDim.x) * p.RG;
    down = false;
    open_gu();
    if (!valid) open_down();
  }

  __device__ __forceinline__ void next() {
    if (!down) {
      if (++kc < nkc) return;
      g += nn;
      open_gu();
      if (!valid) open_down();
      return;
    }
    u0 += ng;
    if (u0 < nU) {
      ng = (nU - u0) < GE ? (nU - u0) : GE;
      return;
    }
    u0 = 0;
    c0 += rc;
    valid = c0 < r1;
    if (valid) {
      rc = (r1 - c0) < RC ? (r1 - c0) : RC;
      ng = nU < GE ? nU : GE;
    }
  }

  __device__ __forceinline__ bool last_kc() const { return kc == nkc - 1; }
  __device__ __forceinline__ bool last_group() const { return u0 + ng >= nU; }
};

// Grid-wide barrier for a cooperative launch: every CTA adds one arrival to a
// 64-bit counter that grows by gridDim.x per launch, then waits (bounded) until
// this launch's arrivals are complete. Called by one thread per CTA.
__device__ __forceinline__ bool grid_barrier(unsigned long long* bar, uint32_t* err) {
  __threadfence();
  const unsigned long long ticket = atomicAdd(bar, 1ull);
  const unsigned long long G = gridDim.x;
  const unsigned long long target = (ticket / G + 1) * G;
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(bar) : "memory");
    if (v >= target) {
      __threadfence();
      return true;
    }
    __nanosleep(32);
  }
  atomicOr(err, kDeviceTimeout);
  return false;
}

template <int KMAX>
__global__ void __launch_bounds__(kFusedThreads, 1) moe_layer_fused_t1(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = p.H, I = p.I, KC = p.KC, S = p.S, nbI = I >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem;
  float4* xs = reinterpret_cast<float4*>(smem + (size_t)S * p.slot_bytes);   // [H/4]
  float4* hs = xs + (H >> 2);                                                  // [k*I/4]
  uint64_t* full = reinterpret_cast<uint64_t*>(hs + ((size_t)p.k * I >> 2));
  uint64_t* empty = full + S;
  uint32_t* sm_words = reinterpret_cast<uint32_t*>(empty + S);                // [16][32]
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kFusedConsumers);
    }
    mbar_init_fence();
  }
  __syncthreads();
  pdl_wait();      // x, topk_ids and topk_w come from upstream work
  pdl_trigger();
  WarpSchedule<KMAX> s;
  s.build(p.ids, 1, p.k, p.E, sm_words + warp * 32, p.err);
  // gate/up stage layout: gate codes, up codes, gate scales, up scales
  const GuStageLayout lay(KC);
  const int o_up = lay.up, o_gs = lay.gs, o_us = lay.us;

  if (warp == kFusedConsumers) {
    // ------------------------------------------------------------ producer
    FusedWalk wk;
    wk.begin(s.n_unique, p);
    int st = 0;
    bool ok = true;
    for (; wk.valid; wk.next(), ++st) {
      const int slot = st % S;
      uint8_t* dst = ring + (size_t)slot * p.slot_bytes;
      int e = 0;
      if (!wk.down) e = s.expert(wk.u);   // warp-collective
      if (lane == 0) {
        if (st >= S) ok = mbar_wait(&empty[slot], ((st / S) - 1) & 1, p.err);
        if (ok && !wk.down) {
          // four tensor copies: the stage's gate rows, up rows, and their scales
          // (full boxes; rows past the expert are never read)
          mbar_expect_tx(&full[slot], 2u * kFusedNeurons * KC + 2u * kFusedNeurons * (KC >> 5));
          const int row = e * 2 * I + wk.i0;
          tma_load_2d(dst, &p.tm_codes, wk.kc * (KC >> 2), row, &full[slot]);
          tma_load_2d(dst + o_up, &p.tm_codes, wk.kc * (KC >> 2), row + I, &full[slot]);
          tma_load_2d(dst + o_gs, &p.tm_scales, wk.kc * (KC >> 7), row, &full[slot]);
          tma_load_2d(dst + o_us, &p.tm_scales, wk.kc * (KC >> 7), row + I, &full[slot]);
        }
      }
      if (wk.down) {
        // one expert id per lane of the group (ng <= GE <= 32)
        int eg = 0;
        for (int gi = 0; gi < wk.ng; ++gi) {
          const int ee = s.expert(wk.u0 + gi);   // warp-collective
          if (lane == gi) eg = ee;
        }
        if (lane == 0 && ok) {
          const uint32_t cb = (uint32_t)wk.rc * I, sb = (uint32_t)wk.rc * nbI;
          mbar_expect_tx(&full[slot], (cb + sb) * wk.ng);
        }
        for (int gi = 0; gi < wk.ng; ++gi) {
          const int ee = __shfl_sync(kFull, eg, gi);
          if (lane == 0 && ok) {
            const uint32_t cb = (uint32_t)wk.rc * I, sb = (uint32_t)wk.rc * nbI;
            const size_t row = (size_t)ee * H + wk.c0;
            uint8_t* d = dst + (size_t)gi * p.EB;
            bulk_copy_g2s(d, p.wd + row * I, cb, &full[slot]);
            bulk_copy_g2s(d + (size_t)p.RC * I, p.sd + row * nbI, sb, &full[slot]);
          }
        }
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (!ok) break;
    }
    // never leave with copies in flight: the last stages' copies must land
    if (lane == 0)
      for (int d = st - 1; d >= 0 && d >= st - S; --d) mbar_wait(&full[d % S], (d / S) & 1, p.err);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = threadIdx.x;                    // consumer thread index
  const int ncons = kFusedConsumers * 32;
  // this lane's routing weight (lane j < k holds w[j]); out-of-range ids give
  // h = 0 (written by the CTA that owns no neuron: CTA 0) and no down term
  const float wj = (lane < p.k) ? __ldg(p.w + lane) : 0.f;
  if (blockIdx.x == 0 && warp == 0 && s.badmask) {
    for (uint32_t m = s.badmask; m; m &= m - 1) {
      uint16_t* row = p.h + (size_t)(__ffs(m) - 1) * I;
      for (int i = 0; i < I; ++i) row[i] = 0;   // lane 0 alone holds the token
    }
  }
  for (int c = ctid; c < (H >> 3); c += ncons) {   // x -> swizzled FP32 pieces
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x) + c);
    const int q = c >> 1, jj = (c & 1) * 2;
    xs[piece_slot(q, jj)] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    xs[piece_slot(q, jj + 1)] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
  }
  named_sync(1, ncons);

  FusedWalk wk;
  wk.begin(s.n_unique, p);
  float ag = 0.f, au = 0.f, acc = 0.f;
  bool barrier_done = false;
  // a warp whose bounded wait gave up stops waiting and computing but still
  // reaches every arrival and named barrier, so no other warp can hang on it
  bool dead = false;
  const int swz = (lane >> 1) & 3;   // piece q = 32 m + lane: (q >> 1) & 3 = (lane >> 1) & 3
  for (int st = 0; wk.valid; wk.next(), ++st) {
    if (wk.down && !barrier_done) {
      // every h value of every CTA is written before any CTA reads h
      named_sync(1, ncons);
      if (ctid == 0) grid_barrier(p.grid_bar, p.err);
      named_sync(1, ncons);
      stage_f32_pieces(p.h, p.k * I, hs, ctid, ncons);
      named_sync(1, ncons);
      barrier_done = true;
    }
    const int slot = st % S;
    if (!dead) dead = !mbar_wait(&full[slot], (st / S) & 1, p.err);
    const uint8_t* base = ring + (size_t)slot * p.slot_bytes;
    if (!wk.down) {
      // ---- gate/up: warp owns neuron i0 + warp over this K-chunk
      if (warp < wk.nn && !dead) {
        const uint8_t* gr = base + warp * KC;
        const uint8_t* ur = base + o_up + warp * KC;
        const uint8_t* gsr = base + o_gs + warp * (KC >> 5);
        const uint8_t* usr = base + o_us + warp * (KC >> 5);
        const int qbase = wk.kc * (KC >> 4);   // first piece of the chunk in the row
#pragma unroll 2
        for (int q = lane; q < (KC >> 4); q += 32) {
          const uint4 gq = *reinterpret_cast<const uint4*>(gr + 16 * q);
          const uint4 uq = *reinterpret_cast<const uint4*>(ur + 16 * q);
          const float scg = ue8m0_to_f32(gsr[q >> 1]);
          const float scu = ue8m0_to_f32(usr[q >> 1]);
          const float4* xp = xs + (size_t)(qbase + q) * 4;
          const float4 x0 = xp[0 ^ swz], x1 = xp[1 ^ swz], x2 = xp[2 ^ swz], x3 = xp[3 ^ swz];
          ag = fmaf(dot16(gq, x0, x1, x2, x3), scg, ag);
          au = fmaf(dot16(uq, x0, x1, x2, x3), scu, au);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (wk.last_kc()) {
        const int e = s.expert(wk.u);   // warp-collective
        if (warp < wk.nn) {
          const float g = warp_sum(ag);
          const float up = warp_sum(au);
          const uint32_t jm = __shfl_sync(kFull, s.jmask(e), 0);
          const uint16_t hb = f32_to_bf16_rn((g / (1.0f + expf(-g))) * up);
          if (lane < p.k && ((jm >> lane) & 1u)) p.h[(size_t)lane * I + wk.i0 + warp] = hb;
        }
        ag = au = 0.f;
      }
    } else {
      // ---- down: warp owns row c0 + warp of the chunk, for ng experts
      for (int gi = 0; gi < wk.ng; ++gi) {
        const int e = s.expert(wk.u0 + gi);
        const uint32_t jm = __shfl_sync(kFull, s.jmask(e), 0);
        const float coef = warp_sum(((jm >> lane) & 1u) ? wj : 0.f);
        const int j0 = __ffs(jm) - 1;
        if (warp < wk.rc && jm != 0u && !dead) {
          const uint8_t* cr = base + (size_t)gi * p.EB + (size_t)warp * I;
          const uint8_t* sr = base + (size_t)gi * p.EB + (size_t)p.RC * I + (size_t)warp * nbI;
          const float4* hr = hs + (size_t)j0 * (I >> 2);
          float part = 0.f;
          for (int q = lane; q < (I >> 4); q += 32) {
            const uint4 wq = *reinterpret_cast<const uint4*>(cr + 16 * q);
            const float sc = ue8m0_to_f32(sr[q >> 1]);
            const int sw = (q >> 1) & 3;
            const float4* hp = hr + (size_t)q * 4;
            part = fmaf(dot16(wq, hp[0 ^ sw], hp[1 ^ sw], hp[2 ^ sw], hp[3 ^ sw]), sc, part);
          }
          acc = fmaf(part, coef, acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (wk.last_group()) {
        const float v = warp_sum(acc);
        if (lane == 0 && warp < wk.rc) p.y[wk.c0 + warp] = f32_to_bf16_rn(v);
        acc = 0.f;
      }
    }
  }
  if (!barrier_done) {
    // a CTA with no down stages still takes part in the grid barrier
    named_sync(1, ncons);
    if (ctid == 0) grid_barrier(p.grid_bar, p.err);
  }
  if (s.n_unique == 0) {
    // no valid expert at all: the CTA's output rows are zero
    for (int r = wk.r0 + ctid; r < wk.r1; r += ncons) p.y[r] = 0;
  }
}

}  // namespace moe
