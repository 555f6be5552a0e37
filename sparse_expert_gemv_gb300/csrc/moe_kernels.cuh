// The decode-layer kernels: router, dedup-schedule export, gate/up, down.
//
// Output-centric throughout (the warp-decode post, cursor.com/blog/warp-decode,
// "What we changed" and "How the two kernels work"): every warp owns output
// scalars, streams the weight rows they need straight from HBM, decodes the
// block-scaled codes in registers, accumulates in private FP32 registers and
// finishes with a shfl.xor butterfly. No warp shares partial sums with
// another. The projection kernels take the weight format (Mxfp8 or Mxfp4) as
// a template argument F; a weight row of K elements is K * F::kBlockBytes / 32
// code bytes.
#pragma once

#include "moe_f16blocks.cuh"

namespace moe {

constexpr int kWarps = 8;               // 8-warp CTAs, as in the pages' gate/up kernel
constexpr int kThreads = kWarps * 32;
constexpr int kMaxTokensPerLaunch = 32; // tokens of one schedule (one per lane)

// ---------------------------------------------------------------------------
// Router: softmax over E logits, top-k (ties to the lower id), renormalise.
// One warp per token; lane l holds logits l, l+32, ...
// ---------------------------------------------------------------------------

template <int RMAX>
__global__ void __launch_bounds__(kThreads) moe_route_topk(const float* __restrict__ logits, int T,
                                                           int E, int k, int32_t* __restrict__ ids,
                                                           float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (t >= T) return;
  float v[RMAX];
  const float* row = logits + (size_t)t * E;
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    const int e = lane + 32 * r;
    v[r] = (e < E) ? __ldg(row + e) : 0.f;
  }
  uint32_t taken = 0;
  float my_v = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float best = -__int_as_float(0x7f800000);
    int bidx = 0x7fffffff;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      const int e = lane + 32 * r;
      if (e < E && !((taken >> r) & 1u) && (v[r] > best || (v[r] == best && e < bidx))) {
        best = v[r];
        bidx = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, best, o);
      const int oi = __shfl_xor_sync(kFull, bidx, o);
      if (ov > best || (ov == best && oi < bidx)) {
        best = ov;
        bidx = oi;
      }
    }
    if ((bidx & 31) == lane) taken |= 1u << (bidx >> 5);
    if (lane == j) {
      my_v = best;
      my_id = bidx;
    }
  }
  const float top = __shfl_sync(kFull, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - top) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = ex / sum;
  }
}

// ---------------------------------------------------------------------------
// Dedup schedule export (one warp, <= 32 tokens): the same WarpSchedule the
// projection kernels build on chip, written out for inspection.
// ---------------------------------------------------------------------------

template <int KMAX>
__global__ void __launch_bounds__(32) moe_dedup_schedule_kernel(const int32_t* __restrict__ ids,
                                                                int T, int k, int E,
                                                                int32_t* uniq, int32_t* offsets,
                                                                int32_t* pairs, int32_t* n_uniq,
                                                                uint32_t* err) {
  __shared__ uint32_t sm_words[32];
  __shared__ uint32_t sm_ids[schedule_id_bytes(KMAX) / 4];
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  WarpSchedule<KMAX, IdStore::kShared> s;
  s.build(ids, T, k, E, sm_words, err, sm_ids);
  int base = 0;
  for (int u = 0; u < s.n_unique; ++u) {
    const int e = s.expert(u);
    const uint32_t jm = s.jmask(e);
    const int cnt = __popc(jm);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    int pos = base + incl - cnt;
    for (uint32_t m = jm; m; m &= m - 1) pairs[pos++] = lane * k + (__ffs(m) - 1);
    if (lane == 0) {
      uniq[u] = e;
      offsets[u] = base;
    }
    base += __shfl_sync(kFull, incl, 31);
  }
  if (lane == 0) {
    offsets[s.n_unique] = base;
    *n_uniq = s.n_unique;
  }
}

// ---------------------------------------------------------------------------
// Gate/up: h[t, j, i] = bf16(SiLU(g) * u) for every token routed to expert e.
//
// Work unit = (unique expert u, neuron i): one warp streams gate row i and up
// row i of expert u once and applies them to up to NT of the expert's tokens
// at a time (more tokens: another pass over the same rows, from L2). Lane l
// takes the 32-element blocks b = l, l+32, ... of the H-long rows, so each
// 256-bit load of a warp covers 1 KB of one row. The block's partial dots are
// scaled by the block's UE8M0 factor and accumulated in FP32 per token.
// ---------------------------------------------------------------------------

struct GateUpParams {
  const uint16_t* x;      // [T, H] bf16
  const int32_t* ids;     // [T, k]
  const uint8_t* wgu;     // [E, 2I, H * F::kBlockBytes / 32]
  const uint8_t* sgu;     // [E, 2I, H/32]
  uint16_t* h;            // [T, k, I] bf16
  uint32_t* err;
  int T, k, E, H, I;
};

template <int NT, class F>
__device__ __forceinline__ void gate_up_block(const uint32_t (&qg)[F::kWords],
                                              const uint32_t (&qu)[F::kWords], float scg,
                                              float scu, const uint16_t* __restrict__ x,
                                              const TokenGroup<NT>& tg, int H, int b,
                                              float (&ag)[NT], float (&au)[NT]) {
  float pg[NT], pu[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) pg[n] = pu[n] = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float g[8], u[8];
    F::chunk_f32(qg, c, g);
    F::chunk_f32(qu, c, u);
    uint32_t gm = tg.grp;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      if (n < tg.nt) {
        const uint4 xv = ld_act16(x + (size_t)tg.token(n, gm) * H + b * 32 + c * 8);
        const float xs[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                             bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          pg[n] = fmaf(g[m], xs[m], pg[n]);
          pu[n] = fmaf(u[m], xs[m], pu[n]);
        }
      }
    }
  }
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    ag[n] = fmaf(pg[n], scg, ag[n]);
    au[n] = fmaf(pu[n], scu, au[n]);
  }
}

template <int NT, int KMAX, class F>
__global__ void __launch_bounds__(kThreads, 2) moe_gate_up_3d_batched(GateUpParams p) {
  __shared__ uint32_t sm_words[kWarps][32];
  constexpr IdStore kIds = kWarpIdStore<NT, KMAX>;
  __shared__ uint32_t sm_ids[kWarps][kIds == IdStore::kShared ? schedule_id_bytes(KMAX) / 4 : 1];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  pdl_wait();      // x and topk_ids come from upstream work
  pdl_trigger();   // the down kernel may start fetching its weights
  WarpSchedule<KMAX, kIds> s;
  s.build(p.ids, p.T, p.k, p.E, sm_words[wid], p.err, sm_ids[wid]);
  const int H = p.H, I = p.I, nb = H >> 5;
  // A slot with an out-of-range id gets no unit; its h slice is defined as zero.
  if (__any_sync(kFull, s.badmask != 0u)) {
    for (int t = blockIdx.x * kWarps + wid; t < p.T; t += gridDim.x * kWarps) {
      const uint32_t bm = __shfl_sync(kFull, s.badmask, t);
      for (uint32_t m = bm; m; m &= m - 1) {
        uint16_t* row = p.h + ((size_t)t * p.k + (__ffs(m) - 1)) * I;
        for (int i = lane; i < I; i += 32) row[i] = 0;
      }
    }
  }
  const long long units = (long long)s.n_unique * I;
  for (long long unit = (long long)blockIdx.x * kWarps + wid; unit < units;
       unit += (long long)gridDim.x * kWarps) {
    const int u = (int)(unit / I);
    const int i = (int)(unit - (long long)u * I);
    const int e = s.expert(u);
    const uint32_t jm = s.jmask(e);
    uint32_t tokens = __ballot_sync(kFull, jm != 0u);
    constexpr int CB = F::kBlockBytes;
    const size_t RB = (size_t)nb * CB;        // code bytes per row
    const size_t row = (size_t)e * 2 * I + i;
    const uint8_t* wg = p.wgu + row * RB;
    const uint8_t* wu = wg + (size_t)I * RB;
    const uint8_t* sg = p.sgu + row * nb;
    const uint8_t* su = sg + (size_t)I * nb;
    while (tokens) {
      TokenGroup<NT> tg;   // this pass's tokens: the lowest NT of `tokens`
      tg.take(tokens);
      const int nt = tg.nt;
      float ag[NT], au[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) ag[n] = au[n] = 0.f;
      // two blocks in flight per lane: issue block b+32 before computing b
      uint32_t qg0[F::kWords], qu0[F::kWords], qg1[F::kWords], qu1[F::kWords];
      uint32_t s0g = 0, s0u = 0, s1g = 0, s1u = 0;
      int b = lane;
      if (b < nb) {
        F::load(wg + b * CB, qg0);
        F::load(wu + b * CB, qu0);
        s0g = ld_scale(sg + b);
        s0u = ld_scale(su + b);
      }
      while (b < nb) {
        const int b1 = b + 32;
        if (b1 < nb) {
          F::load(wg + b1 * CB, qg1);
          F::load(wu + b1 * CB, qu1);
          s1g = ld_scale(sg + b1);
          s1u = ld_scale(su + b1);
        }
        gate_up_block<NT, F>(qg0, qu0, ue8m0_to_f32(s0g), ue8m0_to_f32(s0u), p.x, tg, H, b,
                             ag, au);
        if (b1 >= nb) break;
        const int b2 = b1 + 32;
        if (b2 < nb) {
          F::load(wg + b2 * CB, qg0);
          F::load(wu + b2 * CB, qu0);
          s0g = ld_scale(sg + b2);
          s0u = ld_scale(su + b2);
        }
        gate_up_block<NT, F>(qg1, qu1, ue8m0_to_f32(s1g), ue8m0_to_f32(s1u), p.x, tg, H, b1,
                             ag, au);
        b = b2;
      }
      uint32_t gm = tg.grp;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        if (n < nt) {
          const int t = tg.token(n, gm);
          const float g = warp_sum(ag[n]);
          const float up = warp_sum(au[n]);
          const uint32_t jt = __shfl_sync(kFull, jm, t);
          const float hv = (g / (1.0f + expf(-g))) * up;
          const uint16_t hb = f32_to_bf16_rn(hv);
          if (lane < p.k && ((jt >> lane) & 1u)) p.h[((size_t)t * p.k + lane) * I + i] = hb;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Down: y[t, r] = bf16(sum_j w[t, j] * sum_i dq(Wd[e_j, r, i]) * h[t, j, i]).
//
// One warp per (token t, output row r); a CTA covers 8 consecutive rows of one
// token. The warp's k rows Wd[e_j, r, :] are laid out as k*I/32 blocks of 32
// elements and dealt to the lanes (block f = j*I/32 + b to lane f % 32), so all
// 32 lanes stream even when I/32 < 32; down_load_round fetches one round of
// them. The kernel (moe_down_3d_batched, below) reads h[t] once per CTA into
// shared memory as f16 blocks. With `early` set, the
// first round of weight loads is issued before waiting for the gate/up kernel
// (those rows depend only on topk_ids).
// ---------------------------------------------------------------------------

struct DownParams {
  const uint16_t* h;      // [T, k, I] bf16
  const int32_t* ids;     // [T, k]
  const float* w;         // [T, k]
  const uint8_t* wd;      // [E, H, I * F::kBlockBytes / 32]
  const uint8_t* sd;      // [E, H, I/32]
  uint16_t* y;            // [T, H] bf16
  uint32_t* err;
  int T, k, E, H, I;
  int early;
};

template <int QMAX, class F>
__device__ __forceinline__ void down_load_round(const DownParams& p, int f0, int nf, int nbI, int r,
                                                int id, float wj, uint32_t (&q)[QMAX][F::kWords],
                                                float (&sc)[QMAX], float (&wsel)[QMAX],
                                                bool (&valid)[QMAX]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int qi = 0; qi < QMAX; ++qi) {
    const int f = f0 + lane + 32 * qi;
    const int j = (f < nf) ? f / nbI : 0;
    const int b = f - j * nbI;
    const int e = __shfl_sync(kFull, id, j);
    wsel[qi] = __shfl_sync(kFull, wj, j);
    valid[qi] = (f < nf) && (e >= 0);
    if (valid[qi]) {
      const size_t rowi = (size_t)e * p.H + r;
      F::load(p.wd + (rowi * nbI + b) * F::kBlockBytes, q[qi]);
      sc[qi] = ue8m0_to_f32(ld_scale(p.sd + rowi * nbI + b));
    } else {
#pragma unroll
      for (int m = 0; m < F::kWords; ++m) q[qi][m] = 0u;
      sc[qi] = 0.f;
    }
  }
}

// ---------------------------------------------------------------------------
// Gate/up for several tokens with x staged in shared memory (T >= 2 when the
// T tokens' x fits): the work units and token groups of
// moe_gate_up_3d_batched, but each CTA converts x once to f16 blocks scaled
// by a power of two (as the one-launch kernel does), each weight block is
// decoded once to f16 pairs for all of a group's tokens, and fma.rn.f32.f16
// forms every product (exact, as the header explains).
// ---------------------------------------------------------------------------

constexpr int kXsWarps = 16;
constexpr int kXsThreads = kXsWarps * 32;

// Shared-memory bytes of moe_gate_up_3d_batched_xs for T tokens of H and
// KMAX slots a token (all of it dynamic: the warps' schedule words and id
// tables, then x as f16 blocks, then their factors).
__host__ __device__ constexpr size_t gate_up_xs_ids_offset() { return (size_t)kXsWarps * 32 * 4; }
__host__ __device__ constexpr size_t gate_up_xs_x_offset(int kmax) {
  return gate_up_xs_ids_offset() + (size_t)kXsWarps * schedule_id_bytes(kmax);
}
__host__ __device__ constexpr size_t gate_up_xs_smem(int T, int H, int kmax) {
  return gate_up_xs_x_offset(kmax) + (size_t)T * (H >> 5) * (64 + 4);
}

// D: weight blocks per lane in flight (1, or 2 when registers allow).
template <int NT, int KMAX, class F, int D = 1>
__global__ void __launch_bounds__(kXsThreads, 1) moe_gate_up_3d_batched_xs(GateUpParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int H = p.H, I = p.I, nb = H >> 5;
  uint32_t* sm_words = reinterpret_cast<uint32_t*>(smem);              // [warps][32]
  uint32_t* sm_ids = reinterpret_cast<uint32_t*>(smem + gate_up_xs_ids_offset());
  uint8_t* xs = smem + gate_up_xs_x_offset(KMAX);                      // [T][nb] x blocks
  float* xf = reinterpret_cast<float*>(xs + (size_t)p.T * nb * 64);    // [T][nb] factors
  pdl_wait();      // x and topk_ids come from upstream work
  pdl_trigger();   // the down kernel may start fetching its weights
  WarpSchedule<KMAX, kWarpIdStore<NT, KMAX>> s;   // (the id tables are reserved either way)
  s.load(p.ids, p.T, p.k);
  // x -> f16 blocks while the ids are in flight
#pragma unroll 1
  for (int idx = threadIdx.x; idx < p.T * nb; idx += kXsThreads) {
    const int t = idx / nb, b = idx - t * nb;
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * H) + 4 * b;
    const uint4 v[4] = {__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3)};
    xf[idx] = stage_block_f16(v, xs + 64 * idx, b);
  }
  s.finish(p.E, sm_words + wid * 32, p.err, sm_ids + wid * (schedule_id_bytes(KMAX) / 4));
  // A slot with an out-of-range id gets no unit; its h slice is defined as zero.
  if (__any_sync(kFull, s.badmask != 0u)) {
    for (int t = blockIdx.x * kXsWarps + wid; t < p.T; t += gridDim.x * kXsWarps) {
      const uint32_t bm = __shfl_sync(kFull, s.badmask, t);
      for (uint32_t m = bm; m; m &= m - 1) {
        uint16_t* row = p.h + ((size_t)t * p.k + (__ffs(m) - 1)) * I;
        for (int i = lane; i < I; i += 32) row[i] = 0;
      }
    }
  }
  __syncthreads();   // x staged
  const LaneBlock lb(lane);
  const bool swap = lb.c_first != 0;
  const long long units = (long long)s.n_unique * I;
#pragma unroll 1
  for (long long unit = (long long)blockIdx.x * kXsWarps + wid; unit < units;
       unit += (long long)gridDim.x * kXsWarps) {
    const int u = (int)(unit / I);
    const int i = (int)(unit - (long long)u * I);
    const int e = s.expert(u);
    const uint32_t jm = s.jmask(e);
    uint32_t tokens = __ballot_sync(kFull, jm != 0u);
    constexpr int CB = F::kBlockBytes;
    const size_t RB = (size_t)nb * CB;        // code bytes per row
    const size_t row = (size_t)e * 2 * I + i;
    const uint8_t* wg = p.wgu + row * RB;
    const uint8_t* wu = wg + (size_t)I * RB;
    const uint8_t* sg = p.sgu + row * nb;
    const uint8_t* su = sg + (size_t)I * nb;
#pragma unroll 1
    while (tokens) {
      TokenGroup<NT> tg;   // this pass's tokens: the lowest NT of `tokens`
      tg.take(tokens);
      const int nt = tg.nt;
      float ag[NT], au[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) ag[n] = au[n] = 0.f;
      // the next D blocks' codes are in flight while one is applied
      uint32_t qg[D][F::kWords], qu[D][F::kWords];
      uint32_t s_g[D], s_u[D];
#pragma unroll
      for (int d = 0; d < D; ++d) {
        const int b = lane + 32 * d;
        s_g[d] = s_u[d] = 0;
        if (b < nb) {
          F::load(wg + b * CB, qg[d]);
          F::load(wu + b * CB, qu[d]);
          s_g[d] = ld_scale(sg + b);
          s_u[d] = ld_scale(su + b);
        }
      }
#pragma unroll 1
      for (int b0 = lane; b0 < nb; b0 += 32 * D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
          const int b = b0 + 32 * d;
          if (b < nb) {
            uint32_t whg[16], whu[16];
            F::decode(qg[d], swap, whg);
            F::decode(qu[d], swap, whu);
            const float scg = ue8m0_to_f32(s_g[d]), scu = ue8m0_to_f32(s_u[d]);
            if (b + 32 * D < nb) {
              F::load(wg + (b + 32 * D) * CB, qg[d]);
              F::load(wu + (b + 32 * D) * CB, qu[d]);
              s_g[d] = ld_scale(sg + b + 32 * D);
              s_u[d] = ld_scale(su + b + 32 * D);
            }
            uint32_t gm = tg.grp;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              if (n < nt) {
                const int xb = tg.token(n, gm) * nb + b;
                const uint8_t* act = xs + 64 * xb;
                const float fx = xf[xb];
                ag[n] = fmaf(dot_block_h(whg, act, lb) * fx, scg, ag[n]);
                au[n] = fmaf(dot_block_h(whu, act, lb) * fx, scu, au[n]);
              }
            }
          }
        }
      }
      uint32_t gm = tg.grp;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        if (n < nt) {
          const int t = tg.token(n, gm);
          const float g = warp_sum(ag[n]);
          const float up = warp_sum(au[n]);
          const uint32_t jt = __shfl_sync(kFull, jm, t);
          const uint16_t hb = f32_to_bf16_rn((g / (1.0f + expf(-g))) * up);
          if (lane < p.k && ((jt >> lane) & 1u)) p.h[((size_t)t * p.k + lane) * I + i] = hb;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The down kernel: the work layout above (one warp per (token t, output row
// r), the k rows' 32-element blocks dealt to the lanes, a CTA covering 8 rows
// of one token); h[t] is converted once per CTA to power-of-two-scaled f16
// blocks, keyed by the flat block index f = j * I/32 + b so that lane f % 32
// reads its own swizzle, and each weight block is decoded to f16 pairs for
// fma.rn.f32.f16.
// ---------------------------------------------------------------------------

__host__ __device__ constexpr size_t down_xs_smem(int k, int I) {
  return (size_t)k * (I >> 5) * (64 + 4);
}

template <int QMAX, class F>
__device__ __forceinline__ float down_compute_round_xs(const uint8_t* hs, const float* hfac, int f0,
                                                       const uint32_t (&q)[QMAX][F::kWords],
                                                       const float (&sc)[QMAX],
                                                       const float (&wsel)[QMAX],
                                                       const bool (&valid)[QMAX],
                                                       const LaneBlock& lb, bool swap, float acc) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int qi = 0; qi < QMAX; ++qi) {
    if (valid[qi]) {
      const int f = f0 + lane + 32 * qi;
      uint32_t wh[16];
      F::decode(q[qi], swap, wh);
      const float d = dot_block_h(wh, hs + 64 * f, lb);
      acc = fmaf(d * hfac[f] * sc[qi], wsel[qi], acc);
    }
  }
  return acc;
}

template <int QMAX, class F>
__global__ void __launch_bounds__(kThreads, 2) moe_down_3d_batched(DownParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int t = blockIdx.y;
  const int r = blockIdx.x * kWarps + wid;
  const int k = p.k, I = p.I, nbI = I >> 5, nf = k * nbI;
  uint8_t* hs = smem;                                            // [nf] blocks of 64 B
  float* hfac = reinterpret_cast<float*>(smem + (size_t)nf * 64);  // [nf] factors
  if (!p.early) pdl_wait();
  int id = -1;
  float wj = 0.f;
  if (lane < k) {
    id = __ldg(p.ids + (size_t)t * k + lane);
    wj = __ldg(p.w + (size_t)t * k + lane);
    if (id < 0 || id >= p.E) {
      if (blockIdx.x == 0 && wid == 0) atomicOr(p.err, kDeviceBadId);
      id = -1;
    }
  }
  uint32_t q[QMAX][F::kWords];
  float sc[QMAX], wsel[QMAX];
  bool valid[QMAX];
  down_load_round<QMAX, F>(p, 0, nf, nbI, r, id, wj, q, sc, wsel, valid);
  if (p.early) pdl_wait();   // h is written by the gate/up kernel
  {
    const uint4* ht = reinterpret_cast<const uint4*>(p.h + (size_t)t * k * I);
#pragma unroll 1
    for (int f = threadIdx.x; f < nf; f += kThreads) {
      const uint4* src = ht + 4 * f;
      const uint4 v[4] = {src[0], src[1], src[2], src[3]};
      hfac[f] = stage_block_f16(v, hs + 64 * f, f);
    }
  }
  __syncthreads();
  pdl_trigger();
  const LaneBlock lb(lane);
  const bool swap = lb.c_first != 0;
  float acc = down_compute_round_xs<QMAX, F>(hs, hfac, 0, q, sc, wsel, valid, lb, swap, 0.f);
  for (int f0 = 32 * QMAX; f0 < nf; f0 += 32 * QMAX) {
    down_load_round<QMAX, F>(p, f0, nf, nbI, r, id, wj, q, sc, wsel, valid);
    acc = down_compute_round_xs<QMAX, F>(hs, hfac, f0, q, sc, wsel, valid, lb, swap, acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) p.y[(size_t)t * p.H + r] = f32_to_bf16_rn(acc);
}

}  // namespace moe
