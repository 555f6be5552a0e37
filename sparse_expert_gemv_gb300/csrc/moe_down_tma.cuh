// Down projection for several tokens, with TMA-streamed weight rows.
//
// The warp-decode post (cursor.com/blog/warp-decode, "How the two kernels
// work") gives each warp one output scalar y[t, r] and has it stream row r of
// each of token t's routed experts, accumulate the routing-weighted dot
// products in registers and reduce with a butterfly. That is what the warps
// here do; what changes is how the rows reach them. One producer warp per
// CTA walks the CTA's share of (token t, 16-row tile) items in order and
// streams, for each distinct expert routed to t, that expert's 16 rows of
// W_down (and their scales) into a ring of shared-memory slots with TMA
// tensor copies, as far ahead as the ring allows; 16 consumer warps, one per
// row of the tile, reduce each slot against h[t], which the CTA stages once
// per token as f16 blocks (moe_f16blocks.cuh). A slot arriving, not a launch
// or a load round trip, is what a warp waits for, so the stream stays ahead
// of the arithmetic.
//
// Duplicate ids of a token are one distinct expert whose routing weight is
// the sum of theirs (their h rows are equal); an id outside [0, E) adds
// nothing and sets the error flag.
#pragma once

#include <cuda.h>

#include "moe_kernels.cuh"

namespace moe {

constexpr int kDnConsumers = 16;                        // consumer warps: one row each
constexpr int kDnThreads = (kDnConsumers + 1) * 32;     // + one producer warp
constexpr int kDnRows = 16;                             // rows per tile

struct DownTmaParams {
  // W_down codes as a 4D uint32 tensor [E][H][IB/(4*kin)][kin] with boxes of
  // one expert's 16 rows, and its scales as a 2D uint32 tensor [E][H*I/128]
  // with boxes of 16 rows' scale bytes (IB = code bytes per row)
  CUtensorMap tm_codes;
  CUtensorMap tm_scales;
  const uint16_t* h;      // [T, k, I] bf16
  const int32_t* ids;     // [T, k]
  const float* w;         // [T, k]
  uint16_t* y;            // [T, H] bf16
  uint32_t* err;
  int T, k, E, H, I;
  int SG;                 // ring slots
};

// Shared-memory map (byte offsets, 128-byte aligned): the ring (slot = 16
// rows of codes, then their scales), h[t] as f16 blocks of each distinct
// expert, the blocks' factors times the expert's routing weight, the
// distinct experts' first slot and routing weight, and the mbarriers.
struct DnTmaSmem {
  int slot, codes, hs, hf, dj, dw, bars, total;
  __host__ __device__ DnTmaSmem(int SG, int I, int IB, int k) {
    codes = kDnRows * IB;
    slot = round128(kDnRows * IB + kDnRows * (I >> 5));
    int o = SG * slot;
    hs = o;
    o += round128(k * (I >> 5) * 64);
    hf = o;
    o += round128(k * (I >> 5) * 4);
    dj = o;
    o += round128(k * 4);
    dw = o;
    o += round128(k * 4);
    bars = o;
    o += round128(2 * SG * 8);
    total = o;
  }
};

// A token's distinct valid experts, one per lane j < k that holds the first
// occurrence of its id: the mask of those lanes (ascending j = the order of
// the stream) and this lane's id (-1 if invalid).
struct TokenExperts {
  int id;
  uint32_t first;   // lanes holding a first occurrence
  uint32_t bad;     // lanes holding an out-of-range id
  __device__ __forceinline__ void load(const int32_t* __restrict__ ids, int t, int k, int E) {
    const int lane = threadIdx.x & 31;
    id = lane < k ? __ldg(ids + (size_t)t * k + lane) : -1;
    const bool inv = lane < k && (id < 0 || id >= E);
    if (inv) id = -1;
    bad = __ballot_sync(kFull, inv);
    // first occurrence: no lower lane holds the same valid id
    const uint32_t same = __match_any_sync(kFull, id);
    first = __ballot_sync(kFull, id >= 0 && (same & ((1u << lane) - 1u)) == 0u);
  }
};

template <class F>
__global__ void __launch_bounds__(kDnThreads, 1) moe_down_tma(const __grid_constant__ DownTmaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int CB = F::kBlockBytes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = p.H, I = p.I, k = p.k, SG = p.SG, nbI = I >> 5, IB = nbI * CB;
  const int nrt = H / kDnRows;
  const DnTmaSmem L(SG, I, IB, k);
  uint8_t* ring = smem;
  uint8_t* hs = smem + L.hs;
  float* hf = reinterpret_cast<float*>(smem + L.hf);
  int* dj = reinterpret_cast<int*>(smem + L.dj);
  float* dw = reinterpret_cast<float*>(smem + L.dw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + SG;
  const int ncons = kDnConsumers * 32;
  if (warp == kDnConsumers && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_codes) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_scales) : "memory");
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < SG; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDnConsumers);
    }
    mbar_init_fence();
  }
  __syncthreads();
  pdl_wait();      // h comes from the gate/up kernel, ids and w from upstream work
  pdl_trigger();
  const long long total = (long long)p.T * nrt;
  const int lo = (int)(total * blockIdx.x / gridDim.x);
  const int hi = (int)(total * (blockIdx.x + 1) / gridDim.x);

  if (warp == kDnConsumers) {
    // ------------------------------------------------------------ producer
    RingPos rg(SG);
    int gi = 0, cur_t = -1;
    bool ok = true;
    TokenExperts te;
#pragma unroll 1
    for (int x = lo; ok && x < hi; ++x) {
      const int t = x / nrt, r0 = (x - t * nrt) * kDnRows;
      if (t != cur_t) {
        cur_t = t;
        te.load(p.ids, t, k, p.E);
        if (te.bad != 0u && lane == 0) atomicOr(p.err, kDeviceBadId);
      }
#pragma unroll 1
      for (uint32_t m = te.first; m; m &= m - 1, rg.next(), ++gi) {
        const int e = __shfl_sync(kFull, te.id, __ffs(m) - 1);
        if (lane == 0 && gi >= SG) ok = mbar_wait(&empty[rg.slot], rg.phase ^ 1u, p.err);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* dst = ring + (size_t)rg.slot * L.slot;
          uint64_t* bar = &full[rg.slot];
          mbar_expect_tx(bar, (uint32_t)(kDnRows * IB + kDnRows * nbI));
          tma_load_4d(dst, &p.tm_codes, 0, 0, r0, e, bar);
          tma_load_2d(dst + L.codes, &p.tm_scales, r0 * (nbI >> 2), e, bar);
        }
      }
    }
    // never leave with copies in flight
    if (lane == 0) {
      RingPos r(SG);
      for (int d = 0; d < gi; ++d, r.next())
        if (d >= gi - SG) mbar_wait(&full[r.slot], r.phase, p.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const LaneBlock lb(lane);
  bool dead = false;
  RingPos rg(SG);
  int cur_t = -1, nd = 0;
  TokenExperts te;
#pragma unroll 1
  for (int x = lo; x < hi; ++x) {
    const int t = x / nrt, r0 = (x - t * nrt) * kDnRows;
    if (t != cur_t) {
      // a new token: its distinct experts, and h[t] staged as f16 blocks
      cur_t = t;
      te.load(p.ids, t, k, p.E);
      nd = __popc(te.first);
      named_sync(1, ncons);   // every warp is past its reads of the previous token
      if (warp == 0) {
        const float wj = lane < k ? __ldg(p.w + (size_t)t * k + lane) : 0.f;
        // the routing weight of a distinct expert: its slots' weights summed
        // in slot order
        float c = 0.f;
        for (int j = 0; j < k; ++j) {
          const float wjj = __shfl_sync(kFull, wj, j);
          if (__shfl_sync(kFull, te.id, j) == te.id) c += wjj;
        }
        if ((te.first >> lane) & 1u) {
          const int di = __popc(te.first & ((1u << lane) - 1u));
          dj[di] = lane;
          dw[di] = c;
        }
      }
      named_sync(1, ncons);
#pragma unroll 1
      for (int f = threadIdx.x; f < nd * nbI; f += ncons) {
        const int di = f / nbI, b = f - di * nbI;
        const uint4* src =
            reinterpret_cast<const uint4*>(p.h + ((size_t)t * k + dj[di]) * I) + 4 * b;
        const uint4 v[4] = {src[0], src[1], src[2], src[3]};
        hf[f] = dw[di] * stage_block_f16(v, hs + 64 * f, b);
      }
      named_sync(1, ncons);
    }
    float acc = 0.f;
#pragma unroll 1
    for (int di = 0; di < nd; ++di, rg.next()) {
      if (!dead) dead = !mbar_wait(&full[rg.slot], rg.phase, p.err);
      if (!dead) {
        const uint8_t* st = ring + (size_t)rg.slot * L.slot;
        const uint8_t* row = st + warp * IB;
        const uint8_t* sc = st + L.codes + warp * nbI;
        for (int b = lane; b < nbI; b += 32) {
          const int f = di * nbI + b;
          const float d = F::dot_smem(row + CB * b, hs + 64 * f, lb);
          acc = fmaf(d * ue8m0_to_f32(sc[b]), hf[f], acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[rg.slot]);
    }
    const float v = warp_sum(acc);
    if (lane == 0) p.y[(size_t)t * H + r0 + warp] = f32_to_bf16_rn(v);
  }
}

}  // namespace moe
