// The whole single-token layer in one persistent launch.
//
// Both projections of the warp-decode post (cursor.com/blog/warp-decode, "How
// the two kernels work") run here as two phases of one cooperative kernel with
// one CTA per SM. The split of work is the post's output-centric one: in the
// gate/up phase a warp owns one intermediate neuron and reduces its gate and
// up dot products itself; in the down phase a warp owns one output row.
//
// What the single launch adds is the memory stream. One producer warp per CTA
// streams, with TMA, everything the CTA reads through one ring of SG
// shared-memory slots guarded by mbarriers: first its gate/up tiles (fifteen
// neurons' gate and up rows over a K-chunk), then its down rows for every
// routed expert, in groups of whole slots, each group issued as soon as a
// gate/up stage has freed its slot. HBM so keeps streaming while the
// consumers compute, and the down rows land before h has been exchanged. h
// itself is staged in a region of its own.
//
// Every CTA needs every h value, so the CTAs meet at a grid barrier between
// the phases (the launch is cooperative, so all of them are resident). Each
// CTA learns the launch's index from one counter add at its start; at the
// barrier it then only posts a release add to a second counter and, after
// preparing its down work (where each item's rows sit, the arrival of its
// down groups), polls it (acquire loads) for the value that index implies.
// (Publishing h as epoch-tagged words that readers poll directly measured
// slower on this part: every CTA polling all of h floods L2 while the down
// rows stream.)
//
// Arithmetic. Each lane reduces one 32-element MX block at a time: 32 codes
// (E4M3 for MXFP8, E2M1 for MXFP4: the template argument F) against 32
// activations, FP32 accumulation, then the block's UE8M0 scale. The
// activations (x in the gate/up phase, h in the down phase) are held in
// shared memory as f16 after multiplying each 32-element block by a power of
// two 2^e that brings its largest magnitude into [2^14, 2^15); the factor
// 2^-e is applied to the block's sum. Both code types convert to f16
// exactly, a bf16 value scaled that way is exact in f16 whenever it lies
// within 2^-28 of its block's largest magnitude, and an f16 x f16 product is
// exact in FP32, so fma.rn.f32.f16 gives the same sums as FP32 FMAs on the
// decoded values.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "moe_decode_timeline.h"   // stamp indices of MOE_TIMELINE builds
#include "moe_kernels.cuh"

namespace moe {

// 15 consumer warps + 1 producer warp: 4 warps per SM sub-partition, so each
// thread may hold up to 128 registers (a sub-partition has 16K).
constexpr int kFusedConsumers = 15;                       // consumer warps
constexpr int kFusedThreads = (kFusedConsumers + 1) * 32; // + one producer warp
constexpr int kFusedNeurons = kFusedConsumers;            // gate/up neurons per stage

// Byte counts below: a row of K weights holds K * F::kBlockBytes / 32 code
// bytes (RB for a gate/up row of H, IB for a down row of I, KB for a K-chunk
// of KC).
struct FusedParams {
  // W_gateup codes as a 3D uint32 tensor [E*2I][RB/(4*kin)][kin] with boxes of
  // kFusedNeurons rows x KB bytes, and its scales as a 2D uint32 tensor
  // [E*2I][H/128] with boxes of kFusedNeurons rows x KC/32 scale bytes
  CUtensorMap tm_codes;
  CUtensorMap tm_scales;
  // W_down codes as a 4D uint32 tensor [E][H][IB/(4*kin_d)][kin_d] with boxes
  // of RC rows of one expert, and its scales as a 2D uint32 tensor
  // [E][H*I/128] with boxes of RC rows' scale bytes (rows past H read as zeros)
  CUtensorMap tm_dcodes;
  CUtensorMap tm_dscales;
  const uint16_t* x;          // [1, H] bf16
  const int32_t* ids;         // [1, k]
  const float* w;             // [1, k]
  const uint8_t* wgu;         // [E, 2I, RB]
  const uint8_t* sgu;         // [E, 2I, H/32]
  const uint8_t* wd;          // [E, H, IB]
  const uint8_t* sd;          // [E, H, I/32]
  uint16_t* h;                // [1, k, I] bf16 (written, then read back through L2)
  uint16_t* y;                // [1, H] bf16
  uint32_t* err;
  unsigned long long* launch_ctr;  // grows by gridDim.x per launch, at kernel start
  unsigned long long* bar_ctr;     // grows by gridDim.x per launch, at the grid barrier
  unsigned long long* stamps;      // per-CTA timeline (builds with MOE_TIMELINE), else null
  int k, E, H, I;
  int KC;       // gate/up weights per row per stage (KB = 512, 1024 or 2048 bytes), divides H
  int kin;      // uint32 words per innermost box row of tm_codes (KB/4 or 256)
  int SG;       // gate/up ring slots
  int slot_g;   // bytes per gate/up slot (GuStageLayout(KB, KC).end)
  int SR;       // down row chunks per ring slot (one routed expert's RC rows each)
  int slot_d;   // bytes per down chunk in a slot: RC rows of codes, then RC rows of scales
  int RG;       // down row granule (keeps scale copies 16-byte aligned)
  int RC;       // down rows per chunk (multiple of RG, <= kFusedConsumers)
  int nkc;      // H / KC: K-chunks per gate/up row
  int kdiv;     // KB / (4 * kin): tm_codes dim-1 boxes per K-chunk
  int nrg;      // H / RG: down row granules
};

// Byte offsets of a gate/up stage (KB code bytes and KC/32 scale bytes per
// row) in a ring slot: gate codes, up codes, gate scales, up scales, each
// region starting on a 128-byte boundary (the TMA tensor copies that fill
// them require it); `end` is the bytes used.
struct GuStageLayout {
  int up, gs, us, end;
  __host__ __device__ GuStageLayout(int KB, int KC)
      : up(round128(kFusedNeurons * KB)),
        gs(2 * round128(kFusedNeurons * KB)),
        us(2 * round128(kFusedNeurons * KB) + round128(kFusedNeurons * (KC >> 5))),
        end(2 * round128(kFusedNeurons * KB) + 2 * round128(kFusedNeurons * (KC >> 5))) {}
};

// Shared-memory map of the kernel (byte offsets, each 128-byte aligned). The
// SG ring slots start at 0.
struct FusedSmem {
  int xs;       // x as f16, [H/32] blocks of 64 bytes (swizzled 16-byte chunks)
  int xf;       // [H/32] FP32 block factors 2^-e of x
  int ep;       // the value bar_ctr reaches when this launch's CTAs have all arrived
  int cf;       // [k] combined routing weight of each unique expert
  int jz;       // [k] first slot j routed to each unique expert
  int bars;     // mbarriers: full[SG], empty[SG], then one for the h copy
  int words;    // 16 warps x 32 words of expert bitmap
  // h of each unique expert as f16 ([k][I/32] blocks of 64 bytes); then, per
  // down item t (block t % (I/32) of unique expert t / (I/32)), its FP32
  // factor (routing weight x block factor) and the shared-memory offsets of
  // its codes and scales in the current row chunk (row 0)
  int hs, tf, tc, ts;
  int hraw;     // every unique expert's h row as read (bf16, [k][I])
  int total;
  __host__ __device__ FusedSmem(int SG, int slot_g, int H, int I, int k) {
    int o = SG * slot_g;
    xs = o;
    o += round128(H * 2);
    xf = o;
    o += round128((H >> 5) * 4);
    ep = o;
    o += 128;
    cf = o;
    o += round128(k * 4);
    jz = o;
    o += round128(k * 4);
    bars = o;
    o += round128((2 * SG + 1) * 8);
    words = o;
    o += 16 * 32 * 4;
    hs = o;
    o += round128(k * I * 2);
    tf = o;
    o += round128(k * (I >> 5) * 4);
    tc = o;
    o += round128(k * (I >> 5) * 4);
    ts = o;
    o += round128(k * (I >> 5) * 4);
    hraw = o;
    o += round128(k * I * 2);
    total = o;
  }
};

// The CTA's gate/up stage sequence. The grid is split into one group of
// CTAs per unique expert (gridDim.x >= nU; group sizes differ by at most one)
// and each CTA of a group takes an equal share of that expert's I neurons,
// so no CTA's share straddles two experts; the share is cut into stages of
// 15 neurons (the remainder last), each over K-chunks of KC codes.
// Producer and consumers run the same warp-uniform walk.
struct GuWalk {
  int u, i0, nn, kc, nkc;
  int i_beg, n, nst, st;   // the CTA's share [i_beg, i_beg + n), in nst stages
  bool valid;

  // The CTA's expert group u and share [i_beg, i_beg + n) when nU unique
  // experts are routed. Shape and grid values only: each lane computes it
  // for nU = lane + 1 before the routing is known, and begin() picks the
  // lane of the actual nU.
  struct Share {
    int u, i_beg, n;
  };
  __device__ __forceinline__ static Share share(int nU, int I) {
    const uint32_t G = gridDim.x, bx = blockIdx.x;
    Share sh;
    sh.u = (int)(bx * (uint32_t)nU / G);
    const uint32_t lo = ((uint32_t)sh.u * G + nU - 1) / nU;         // first CTA of group u
    const uint32_t hi = ((uint32_t)(sh.u + 1) * G + nU - 1) / nU;   // one past its last
    const uint32_t c = hi - lo, r = bx - lo;
    sh.i_beg = (int)((uint32_t)I * r / c);
    sh.n = (int)((uint32_t)I * (r + 1) / c) - sh.i_beg;
    return sh;
  }

  __device__ __forceinline__ void set_stage() {
    valid = st < nst;
    if (!valid) return;
    // full 15-neuron stages, the remainder last (a stage's TMA box is 15 rows
    // whatever its size, so equal smaller stages would fetch overlapping rows)
    i0 = i_beg + st * kFusedNeurons;
    nn = n - st * kFusedNeurons < kFusedNeurons ? n - st * kFusedNeurons : kFusedNeurons;
  }
  // Warp-collective: `mine` is this lane's share(lane + 1, I).
  __device__ __forceinline__ void begin(int nU, const Share& mine, const FusedParams& p) {
    nkc = p.nkc;
    kc = 0;
    st = 0;
    nst = 0;
    valid = false;
    if (nU <= 0) return;
    u = __shfl_sync(kFull, mine.u, nU - 1);
    i_beg = __shfl_sync(kFull, mine.i_beg, nU - 1);
    n = __shfl_sync(kFull, mine.n, nU - 1);
    nst = (n + kFusedNeurons - 1) / kFusedNeurons;
    set_stage();
  }
  __device__ __forceinline__ void next() {
    if (++kc < nkc) return;
    kc = 0;
    ++st;
    set_stage();
  }
  __device__ __forceinline__ bool last_kc() const { return kc == nkc - 1; }
};

// The CTA's down work: output rows [r0, r1) (whole granules of RG rows), cut
// in chunks of RC rows; each chunk's unique experts in groups of up to SR,
// one group per ring slot.
struct DownWalk {
  int r0, r1, c0, rc, u0, ng, nU, RC, SR;
  bool valid;

  // The CTA's rows (grid values only, so known before the routing).
  __device__ __forceinline__ void rows(const FusedParams& p) {
    const uint32_t nrg = (uint32_t)p.nrg;
    r0 = (int)(nrg * blockIdx.x / gridDim.x) * p.RG;
    r1 = (int)(nrg * (blockIdx.x + 1) / gridDim.x) * p.RG;
  }
  // After rows().
  __device__ __forceinline__ void begin(int nU_, const FusedParams& p) {
    nU = nU_;
    RC = p.RC;
    SR = p.SR;
    c0 = r0;
    u0 = 0;
    valid = r0 < r1 && nU > 0;
    rc = (r1 - c0) < RC ? (r1 - c0) : RC;
    ng = nU < SR ? nU : SR;
  }
  __device__ __forceinline__ void next() {
    u0 += ng;
    if (u0 >= nU) {
      u0 = 0;
      c0 += rc;
      valid = c0 < r1;
      rc = (r1 - c0) < RC ? (r1 - c0) : RC;
    }
    ng = (nU - u0) < SR ? (nU - u0) : SR;
  }
  __device__ __forceinline__ bool last_group() const { return u0 + ng >= nU; }
};

// Grid barrier of a cooperative launch, in two halves used by one thread per
// CTA. Arrival, after the CTA's threads have met at a named barrier: a release
// add of one (cumulative over what those threads wrote). Wait: bounded acquire
// polls until the count reaches this launch's target; false after a timeout
// (with the error flag set).
__device__ __forceinline__ void grid_arrive(unsigned long long* bar) {
  asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(bar) : "memory");
}
__device__ __forceinline__ bool grid_wait(const unsigned long long* bar, unsigned long long target,
                                          uint32_t* err) {
#pragma unroll 1
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(bar) : "memory");
    if (v >= target) return true;
  }
  atomicOr(err, kDeviceTimeout);
  return false;
}

#ifdef MOE_TIMELINE
// Per-CTA timeline: the GPU's global nanosecond timer at the phases of
// moe_decode_timeline.h, MOE_TL_STAMPS words per CTA.
#define MOE_STAMP(i)                                                              \
  do {                                                                            \
    if (p.stamps) {                                                               \
      unsigned long long t_;                                                      \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                      \
      p.stamps[(size_t)blockIdx.x * MOE_TL_STAMPS + (i)] = t_;                    \
    }                                                                             \
  } while (0)
#else
#define MOE_STAMP(i) \
  do {               \
  } while (0)
#endif

template <int KMAX, class F>
__global__ void __launch_bounds__(kFusedThreads, 1) moe_layer_fused_t1(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int CB = F::kBlockBytes;
  const int H = p.H, I = p.I, KC = p.KC, SG = p.SG, nbI = I >> 5;
  const int KB = (KC >> 5) * CB, IB = nbI * CB;   // code bytes of a K-chunk, of a down row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const FusedSmem L(SG, p.slot_g, H, I, p.k);
  uint8_t* ring_g = smem;
  uint8_t* xs = smem + L.xs;
  float* xf = reinterpret_cast<float*>(smem + L.xf);
  unsigned long long* bar_target = reinterpret_cast<unsigned long long*>(smem + L.ep);
  float* cf = reinterpret_cast<float*>(smem + L.cf);
  int* jz = reinterpret_cast<int*>(smem + L.jz);
  uint64_t* full_g = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty_g = full_g + SG;
  uint64_t* full_h = empty_g + SG;     // the h rows' copy
  uint32_t* sm_words = reinterpret_cast<uint32_t*>(smem + L.words);
  const int ctid = threadIdx.x;                    // consumer thread index
  const int ncons = kFusedConsumers * 32;
  if (threadIdx.x == 0) MOE_STAMP(MOE_TL_ENTRY);
  if (warp == kFusedConsumers && lane == 0) {
    // the tensor maps are kernel parameters: fetch them while upstream work drains
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_codes) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_scales) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_dcodes) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_dscales) : "memory");
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < SG; ++i) {
      mbar_init(&full_g[i], 1);
      mbar_init(&empty_g[i], kFusedConsumers);
    }
    mbar_init(full_h, 1);
    mbar_init_fence();
  }
  __syncthreads();
  pdl_wait();      // x, topk_ids and topk_w come from upstream work
  if (threadIdx.x == 0) MOE_STAMP(MOE_TL_INPUTS);
  // the routing first: every warp builds the expert schedule itself
  WarpSchedule<KMAX> s;
  s.load(p.ids, 1, p.k);
  if (warp == kFusedConsumers - 1 && lane == 0) {
    // this launch's index: launches are stream-ordered (and programmatic
    // dependents wait above for the previous one), so each adds gridDim.x
    const unsigned long long ticket = atomicAdd(p.launch_ctr, 1ull);
    *bar_target = (ticket / gridDim.x + 1ull) * gridDim.x;
  }
  // slot j's routing weight in lane j of warp 0, loaded before the stream starts
  const float wj = (warp == 0 && lane < p.k) ? __ldg(p.w + lane) : 0.f;
  if (warp < kFusedConsumers) {
    // x -> f16 blocks first: these loads go out before the weight stream
    #pragma unroll 1
    for (int b = ctid; b < (H >> 5); b += ncons) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x) + 4 * b;
      const uint4 v[4] = {__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3)};
      xf[b] = stage_block_f16(v, xs + 64 * b, b);
    }
  }
  // the stage walks' grid arithmetic while the ids are in flight
  const GuWalk::Share share = GuWalk::share(lane + 1, I);
  DownWalk dw;
  dw.rows(p);
  s.finish(p.E, sm_words + warp * 32, p.err);
  if (warp == kFusedConsumers && lane == 0) MOE_STAMP(MOE_TL_ROUTED);
  const int nU = s.n_unique;
  const GuStageLayout lay(KB, KC);

  if (warp == kFusedConsumers) {
    // ------------------------------------------------------------ producer
    // one ring for everything the CTA streams: its gate/up tiles, then its
    // down row groups, each into the next slot as soon as it is free
    GuWalk gw;
    gw.begin(nU, share, p);
    dw.begin(nU, p);
    RingPos rg(SG);
    int gi = 0;
    bool ok = true;
    #pragma unroll 1
    for (; gw.valid || dw.valid; rg.next(), ++gi) {
      if (lane == 0 && gi >= SG) ok = mbar_wait(&empty_g[rg.slot], rg.phase ^ 1u, p.err);
      ok = __shfl_sync(kFull, ok, 0);
      if (!ok) break;
      uint8_t* dst = ring_g + (size_t)rg.slot * p.slot_g;
      uint64_t* bar = &full_g[rg.slot];
      if (gw.valid) {
        const int e = s.expert(gw.u);   // warp-collective
        if (lane == 0) {
          if (gi == 0) MOE_STAMP(MOE_TL_FIRST_ISSUE);
          // four tensor copies: the stage's gate rows, up rows, and their
          // scales (full boxes; rows past the expert are never read)
          mbar_expect_tx(bar, 2u * kFusedNeurons * KB + 2u * kFusedNeurons * (KC >> 5));
          const int row = e * 2 * I + gw.i0;
          const int kchunk = gw.kc * p.kdiv;
          tma_load_3d(dst, &p.tm_codes, 0, kchunk, row, bar);
          tma_load_3d(dst + lay.up, &p.tm_codes, 0, kchunk, row + I, bar);
          tma_load_2d(dst + lay.gs, &p.tm_scales, gw.kc * (KC >> 7), row, bar);
          tma_load_2d(dst + lay.us, &p.tm_scales, gw.kc * (KC >> 7), row + I, bar);
        }
        gw.next();
      } else {
        // a down group: two tensor copies per expert, RC rows of codes and
        // their scales (full boxes: rows of the next chunk, or zeros past H,
        // are never read)
        if (lane == 0) mbar_expect_tx(bar, (uint32_t)p.RC * (IB + nbI) * dw.ng);
        #pragma unroll 1
        for (int ui = 0; ui < dw.ng; ++ui) {
          const int e = s.expert(dw.u0 + ui);   // warp-collective
          if (lane == 0) {
            uint8_t* d = dst + (size_t)ui * p.slot_d;
            tma_load_4d(d, &p.tm_dcodes, 0, 0, dw.c0, e, bar);
            tma_load_2d(d + (size_t)p.RC * IB, &p.tm_dscales, dw.c0 * (nbI >> 2), e, bar);
          }
        }
        dw.next();
      }
    }
    if (lane == 0) MOE_STAMP(MOE_TL_ISSUE_DONE);
    // the next launch may start its setup (off this warp's critical path)
    pdl_trigger();
    // never leave with copies in flight
    if (lane == 0) {
      RingPos r(SG);
      for (int d = 0; d < gi; ++d, r.next())
        if (d >= gi - SG) mbar_wait(&full_g[r.slot], r.phase, p.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  named_sync(1, ncons);   // x staged
  pdl_trigger();

  if (warp == 0) {
    // while the first tiles are in flight: per unique expert u (lane u), the
    // combined routing weight of its slots and the first slot routed to it
    // (its h row); out-of-range ids give h = 0 (written by CTA 0) and no down
    // term
    const int e = s.expert_per_lane(lane);
    uint32_t jm = 0;
    float c = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const int idj = __shfl_sync(kFull, s.idj(j), 0);   // lane 0 holds the token
      const float wjj = __shfl_sync(kFull, wj, j);
      if (j < p.k && idj == e) {
        jm |= 1u << j;
        c += wjj;
      }
    }
    if (lane < nU) {
      cf[lane] = c;
      jz[lane] = __ffs(jm) - 1;
    }
    if (blockIdx.x == 0) {
      const uint32_t bad = __shfl_sync(kFull, s.badmask, 0);
      for (uint32_t m = bad; m; m &= m - 1) {
        uint16_t* row = p.h + (size_t)(__ffs(m) - 1) * I;
        for (int i = lane; i < I; i += 32) row[i] = 0;
      }
    }
  }

  const LaneBlock lb(lane);
  // a warp whose bounded wait gave up stops waiting and computing but still
  // reaches every arrival and named barrier, so no other warp can hang on it
  bool dead = false;

  // ---- gate/up: warp owns neuron i0 + warp of each stage, lane owns block lane
  RingPos rg(SG);
  {
    GuWalk gw;
    gw.begin(nU, share, p);
    float ag = 0.f, au = 0.f;
    const int nbk = KC >> 5;                      // blocks per row per stage
    #pragma unroll 1
    for (; gw.valid; gw.next(), rg.next()) {
      if (!dead) dead = !mbar_wait(&full_g[rg.slot], rg.phase, p.err);
      if (threadIdx.x == 0 && gw.st == 0 && gw.kc == 0) MOE_STAMP(MOE_TL_FIRST_LANDED);
      if (warp < gw.nn && !dead) {
        const uint8_t* base = ring_g + (size_t)rg.slot * p.slot_g;
        #pragma unroll 1
        for (int bl = lane; bl < nbk; bl += 32) {
          const int b = gw.kc * nbk + bl;         // block of the H row
          const uint8_t* act = xs + 64 * b;
          const float fx = xf[b];
          const float dg = F::dot_smem(base + warp * KB + CB * bl, act, lb);
          const float du = F::dot_smem(base + lay.up + warp * KB + CB * bl, act, lb);
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

  uint8_t* hs = smem + L.hs;
  float* tf = reinterpret_cast<float*>(smem + L.tf);
  int* tc = reinterpret_cast<int*>(smem + L.tc);
  int* ts = reinterpret_cast<int*>(smem + L.ts);

  // ---- down, one row chunk at a time: its groups sit in the ring slots
  // after the gate/up tiles; warp owns row c0 + warp and its lanes take the
  // chunk's items (expert u, block b), two at a time
  dw.begin(nU, p);
  const int n_items = nU * nbI;
  int c0 = 0, rc = 0, ngr = 0;
  RingPos pos0 = rg;
  // The next chunk: where each item's codes and scales sit (expert u's rows
  // are chunk u % SR of the chunk's group u / SR, at ring position
  // pos0 + u / SR) ...
  auto chunk_tables = [&]() {
    c0 = dw.c0;
    rc = dw.rc;
    pos0 = rg;
    #pragma unroll 1
    for (int t = ctid; t < n_items; t += ncons) {
      const int u = t / nbI, b = t - u * nbI;
      const int g = u / p.SR;
      const int slot = pos0.slot + g < SG ? pos0.slot + g : pos0.slot + g - SG;
      const int off = slot * p.slot_g + (u - g * p.SR) * p.slot_d;
      tc[t] = off + CB * b;
      ts[t] = off + p.RC * IB + b;
    }
  };
  // ... and the arrival of its groups
  auto chunk_wait = [&]() {
    ngr = 0;
    #pragma unroll 1
    for (bool more = true; more; rg.next(), ++ngr) {
      if (!dead) dead = !mbar_wait(&full_g[rg.slot], rg.phase, p.err);
      more = !dw.last_group();
      dw.next();
    }
  };
  bool have = dw.valid;
  // every h value of every CTA is written before any CTA reads h; the first
  // chunk is prepared while the other CTAs arrive
  if (ctid == 0) MOE_STAMP(MOE_TL_GATE_UP_DONE);
  named_sync(1, ncons);
  if (ctid == 0) {
    MOE_STAMP(MOE_TL_ARRIVING);
    grid_arrive(p.bar_ctr);
  }
  if (have) {
    chunk_tables();
    chunk_wait();
  }
  if (ctid == 0) {
    MOE_STAMP(MOE_TL_DOWN_LANDED);
    if (!grid_wait(p.bar_ctr, *bar_target, p.err)) dead = true;
    MOE_STAMP(MOE_TL_BARRIER);
    // every unique expert's h row, one bulk copy each (the async proxy reads
    // what other CTAs' generic stores wrote: fence between the proxies)
    asm volatile("fence.proxy.async.global;" ::: "memory");
    mbar_expect_tx(full_h, (uint32_t)(nU * I * 2));
    for (int u = 0; u < nU; ++u)
      bulk_copy_g2s(smem + L.hraw + (size_t)u * I * 2, p.h + (size_t)jz[u] * I, (uint32_t)(I * 2), full_h);
  }
  if (nU > 0 && !dead) dead = !mbar_wait(full_h, 0, p.err);
  // h -> f16 blocks, and each block's factor times its expert's routing weight
  #pragma unroll 1
  for (int t = ctid; t < n_items; t += ncons) {
    const int u = t / nbI, b = t - u * nbI;
    const uint4* src = reinterpret_cast<const uint4*>(smem + L.hraw + (size_t)u * I * 2) + 4 * b;
    const uint4 v[4] = {src[0], src[1], src[2], src[3]};
    tf[t] = cf[u] * stage_block_f16(v, hs + 64 * t, b);
  }
  named_sync(1, ncons);   // h staged
  if (ctid == 0) MOE_STAMP(MOE_TL_H_STAGED);
  {
    // Row pairs over warps: warp w reduces rows q and q + np of the chunk
    // (q = w mod np, np = half the chunk's rows, rounded up) against one
    // half of the items (w / np), so each lane reads an item's h block once
    // for two rows; the two halves' row sums are added in a fixed order.
    float* red = reinterpret_cast<float*>(sm_words);   // [2][16]; the bitmaps are dead
    #pragma unroll 1
    while (have) {
      const int np = (rc + 1) >> 1;
      const int nh = kFusedConsumers / np >= 2 ? 2 : 1;
      const int q = warp % np, hf = warp / np;
      const int ra = q, rb = q + np < rc ? q + np : q;   // no second row: row q again
      float acc_a = 0.f, acc_b = 0.f;
      if (hf < nh && !dead) {
        const int oa = ra * IB, ob = rb * IB, sa = ra * nbI, sb = rb * nbI;
#pragma unroll 1
        for (int t = lane + 32 * hf; t < n_items; t += 32 * nh) {
          float da, db;
          F::dot2_smem(smem + tc[t] + oa, smem + tc[t] + ob, hs + 64 * t, lb, da, db);
          const float f = tf[t];
          acc_a = fmaf(da * ue8m0_to_f32(smem[ts[t] + sa]), f, acc_a);
          acc_b = fmaf(db * ue8m0_to_f32(smem[ts[t] + sb]), f, acc_b);
        }
      }
      const float va = warp_sum(acc_a), vb = warp_sum(acc_b);
      if (lane == 0 && hf < nh) {
        red[hf * 16 + ra] = va;
        if (q + np < rc) red[hf * 16 + q + np] = vb;
      }
      // the chunk's slots are free again
      __syncwarp();
      RingPos r = pos0;
      for (int i = 0; i < ngr; ++i, r.next())
        if (lane == 0) mbar_arrive(&empty_g[r.slot]);
      named_sync(1, ncons);   // every row sum is in red (and the item tables are read)
      if (ctid < rc) {
        float v = red[ctid];
        if (nh == 2) v += red[16 + ctid];
        p.y[c0 + ctid] = f32_to_bf16_rn(v);
      }
      have = dw.valid;
      if (have) {
        chunk_tables();
        chunk_wait();
        // the tables are ready, and red is read before it is written again
        named_sync(1, ncons);
      }
    }
    if (nU == 0) {
      // no valid expert at all: the CTA's output rows are zero
      for (int r = dw.r0 + ctid; r < dw.r1; r += ncons) p.y[r] = 0;
    }
  }
  if (ctid == 0) MOE_STAMP(MOE_TL_DOWN_DONE);
}

}  // namespace moe
