// Down projection for several tokens, each unique expert's rows streamed
// once, products on the tensor cores' warp-level MMA.
//
// y[t, r] = sum over token t's routed experts e of w[t, e] * (W_down[e, r, :]
// . h[t, e, :]) (the warp-decode post, cursor.com/blog/warp-decode, "How the
// two kernels work"). Ordered expert by expert instead of token by token,
// a tile of 16 output rows of one unique expert meets every token routed to
// that expert: a 16 x I by I x (tokens) product. Here one CTA owns a tile of
// 16 output rows and walks the unique experts of the step (their tokens in
// passes of eight). A producer warp streams each expert's 16 rows (codes and
// scales, one TMA tensor copy each) and the h rows of the pass's tokens (one
// bulk copy each) into a ring of shared-memory slots, one (expert, pass) item
// per slot. Consumer warp w owns ring slot w and takes every item that
// lands there, so as many items as the ring holds are reduced at once, no
// warp waits for another, and each slot has one reader that waits for its
// fills in order (a parity wait cannot tell fills two apart). A warp forms its item's products over all of I with mma.sync
// m16n8k16, 32-element block by block (A = the rows' codes decoded to f16,
// exact; B = the tokens' h block converted in registers to f16 after a
// power-of-two scaling that brings the block's largest magnitude into
// [2^14, 2^15), as the other kernels stage activations; FP32 accumulation),
// scales each block's sum by the block's weight scale and activation factor
// in FP32, and adds the item's sums times the routing weight to its own
// accumulator of y[t, tile rows]. When the CTA has walked every expert, the
// 16 warps' accumulators are added in warp order and the CTA writes its rows
// of y for every token. No other CTA touches those rows and nothing is added
// atomically, so the result is reproducible bit for bit.
//
// Duplicate ids of a token are one (token, expert) column whose routing
// weight is the sum of theirs (their h rows are equal); an id outside [0, E)
// adds nothing (the gate/up kernel of the same schedule flags it).
#pragma once

#include <cuda.h>

#include "moe_gate_up_mma.cuh"

namespace moe {

constexpr int kDmConsumers = 16;                        // consumer warps
constexpr int kDmThreads = (kDmConsumers + 1) * 32;     // + one producer warp
constexpr int kDmRows = 16;                             // output rows per tile (the MMA's M)
constexpr int kDmTokens = 8;                            // tokens per pass (the MMA's N)

struct DownMmaParams {
  // W_down codes as a 4D uint32 tensor [E][H][IB/(4*kin)][kin] with boxes of
  // one expert's 16 rows (IB = code bytes per row, at most 1024), and its
  // scales as a 2D uint32 tensor [E][H*I/128] with boxes of 16 rows' scale
  // bytes
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

// Bytes between two tokens' h rows in a slot: I bf16 values plus 16, so that
// the 16-byte loads of eight tokens fall in different bank groups.
__host__ __device__ constexpr int dm_hrow(int I) { return I * 2 + 16; }

// Shared-memory map (byte offsets, 128-byte aligned): the ring (slot = 16
// rows of codes, their scales, eight h rows), each consumer warp's y
// accumulator [T][16], the mbarriers, the warps' schedule words and id
// tables (KMAX slots a token), each warp's column list, the item prefixes,
// and the tokens' routing weights [T][k].
struct DmSmem {
  int codes, hsl, slot, yacc, bars, words, ids, tl, pref, wts, total;
  __host__ __device__ DmSmem(int SG, int I, int IB, int T, int nU_max, int kmax) {
    codes = kDmRows * IB;
    hsl = round128(kDmRows * IB + kDmRows * (I >> 5));
    slot = round128(hsl + kDmTokens * dm_hrow(I));
    int o = SG * slot;
    yacc = o;
    o += round128(kDmConsumers * T * kDmRows * 4);
    bars = o;
    o += round128(2 * SG * 8);
    words = o;
    o += (kDmConsumers + 1) * 32 * 4;
    ids = o;
    o += (kDmConsumers + 1) * schedule_id_bytes(kmax);
    tl = o;
    o += (kDmConsumers + 1) * 3 * kDmTokens * 4;
    pref = o;
    o += round128((nU_max + 1) * 4);
    wts = o;
    o += round128(T * kmax * 4);
    total = o;
  }
};

// Eight bf16 values (one uint4) of a 32-element block whose other 24 values
// sit in the three other lanes of this lane's quad -> four f16x2 words of the
// values times 2^e, e bringing the block's largest magnitude into
// [2^14, 2^15); returns 2^-e. (The scaling of stage_block_f16, one quad
// holding the block.)
__device__ __forceinline__ float quad_block_f16(const uint4 v, uint32_t (&o)[4]) {
  const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(ww[i] & 0x7fffu, (ww[i] >> 16) & 0x7fffu));
  m = max(m, __shfl_xor_sync(kFull, m, 1));
  m = max(m, __shfl_xor_sync(kFull, m, 2));
  const int e = min(141 - (int)(m >> 7), 127);
  const float up = exp2i(e);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 hh = __floats2half2_rn(bf16_lo(ww[i]) * up, bf16_hi(ww[i]) * up);
    o[i] = *reinterpret_cast<const uint32_t*>(&hh);
  }
  return exp2i(-e);
}

template <int KMAX, class F>
__global__ void __launch_bounds__(kDmThreads, 1) moe_down_mma(const __grid_constant__ DownMmaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int CB = F::kBlockBytes, LB = F::kLaneBytes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int H = p.H, I = p.I, k = p.k, SG = p.SG, nbI = I >> 5, IB = nbI * CB;
  const int hrow = dm_hrow(I);
  const int nU_max = min(p.E, p.T * k);
  const DmSmem L(SG, I, IB, p.T, nU_max, KMAX);
  uint8_t* ring = smem;
  float* yacc = reinterpret_cast<float*>(smem + L.yacc);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + SG;
  uint32_t* sm_words = reinterpret_cast<uint32_t*>(smem + L.words);
  int* pref = reinterpret_cast<int*>(smem + L.pref);
  const int ncons = kDmConsumers * 32;
  if (warp == kDmConsumers && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_codes) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_scales) : "memory");
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < SG; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init_fence();
  }
  pdl_wait();      // h comes from the gate/up kernel, ids and w from upstream work
  pdl_trigger();
  WarpSchedule<KMAX, IdStore::kShared> s;
  s.build(p.ids, p.T, k, p.E, sm_words + warp * 32, p.err,
          reinterpret_cast<uint32_t*>(smem + L.ids + warp * schedule_id_bytes(KMAX)));
  const int nU = s.n_unique;
  // the tokens' routing weights, read once per CTA
  float* wts = reinterpret_cast<float*>(smem + L.wts);
  for (int i = threadIdx.x; i < p.T * k; i += kDmThreads) wts[i] = __ldg(p.w + i);
  // passes of each unique expert (its tokens in groups of eight)
#pragma unroll 1
  for (int u = warp; u < nU; u += kDmConsumers + 1) {
    const int n = __popc(__ballot_sync(kFull, s.jmask(s.expert(u)) != 0u));
    if (lane == 0) pref[u + 1] = (n + kDmTokens - 1) / kDmTokens;
  }
  __syncthreads();   // pass counts written
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) pref[0] = 0;
    for (int base = 1; base <= nU; base += 32) {
      const int i = base + lane;
      int v = i <= nU ? pref[i] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
      }
      if (i <= nU) pref[i] = carry + v;
      carry += __shfl_sync(kFull, v, 31);
    }
  }
  __syncthreads();   // prefixes written
  const int nitems = pref[nU];
  const int ntiles = H / kDmRows;
  // this warp's column list of the current item: tokens, their first slot of
  // the expert, their routing weight for it
  int* tl = reinterpret_cast<int*>(smem + L.tl) + warp * 3 * kDmTokens;
  int* tjf = tl + kDmTokens;
  float* tw = reinterpret_cast<float*>(tl + 2 * kDmTokens);

  // The walk over items (expert u, pass) of each tile, shared by producer and
  // consumers: the columns of an item are tokens base .. base+nt-1 of the
  // expert, base = 8 * pass.
  auto columns = [&](int u, int pass, int& e, int& nt) {
    e = s.expert(u);
    const uint32_t jm = s.jmask(e);
    const uint32_t tokens = __ballot_sync(kFull, jm != 0u);
    const int base = kDmTokens * pass;
    nt = min(kDmTokens, __popc(tokens) - base);
    const int rank = __popc(tokens & ((1u << lane) - 1u)) - base;
    float cw = 0.f;   // token `lane`'s weights of its slots on e, in slot order
    for (uint32_t m = jm; m; m &= m - 1) cw += wts[lane * k + __ffs(m) - 1];
    __syncwarp();
    if (jm != 0u && rank >= 0 && rank < kDmTokens) {
      tl[rank] = lane;
      tjf[rank] = __ffs(jm) - 1;
      tw[rank] = cw;
    }
    __syncwarp();
  };

  if (warp == kDmConsumers) {
    // ------------------------------------------------------------ producer
    RingPos rg(SG);
    int gi = 0;
    bool ok = true;
#pragma unroll 1
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      const int r0 = tile * kDmRows;
      int u = 0, pass = 0;
#pragma unroll 1
      for (int it = 0; it < nitems; ++it, rg.next(), ++gi) {
        while (pref[u + 1] - pref[u] <= pass) {
          ++u;
          pass = 0;
        }
        int e, nt;
        columns(u, pass, e, nt);
        ++pass;
        if (lane == 0 && gi >= SG) ok = mbar_wait(&empty[rg.slot], rg.phase ^ 1u, p.err);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* dst = ring + (size_t)rg.slot * L.slot;
          uint64_t* bar = &full[rg.slot];
          mbar_expect_tx(bar, (uint32_t)(kDmRows * IB + kDmRows * nbI + nt * I * 2));
          tma_load_4d(dst, &p.tm_codes, 0, 0, r0, e, bar);
          tma_load_2d(dst + L.codes, &p.tm_scales, r0 * (nbI >> 2), e, bar);
          for (int col = 0; col < nt; ++col)
            bulk_copy_g2s(dst + L.hsl + col * hrow, p.h + ((size_t)tl[col] * k + tjf[col]) * I,
                          (uint32_t)(I * 2), bar);
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
  // item q of the CTA's sequence (all tiles) sits in slot q % SG and is
  // reduced by warp q % SG (warps from SG on have no items)
  bool dead = false;
  float* yw = yacc + warp * p.T * kDmRows;     // this warp's accumulator [T][16]
  int q0 = 0;                                  // sequence number of the tile's first item
#pragma unroll 1
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, q0 += nitems) {
    const int r0 = tile * kDmRows;
    for (int i = lane; i < p.T * kDmRows; i += 32) yw[i] = 0.f;
    __syncwarp();
    int u = 0, pass = 0;
#pragma unroll 1
    for (int it = 0; it < nitems; ++it) {
      while (pref[u + 1] - pref[u] <= pass) {
        ++u;
        pass = 0;
      }
      const int cu = u, cp = pass;
      ++pass;
      const int qi = q0 + it, slot = qi % SG;
      if (slot != warp) continue;
      int e, nt;
      columns(cu, cp, e, nt);
      const uint32_t phase = (uint32_t)((qi / SG) & 1);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (!dead) dead = !mbar_wait(&full[slot], phase, p.err);
      // the shuffles and MMAs below need the whole warp: a wait that ran out
      // on any lane stops them on every lane
      dead = __any_sync(kFull, dead);
      if (!dead) {
        const uint8_t* st = ring + (size_t)slot * L.slot;
        const uint8_t* hb = st + L.hsl + g * hrow + 16 * c;
        const bool tg = g < nt;
#pragma unroll 2
        for (int b = 0; b < nbI; ++b) {
          const uint8_t* cr = st + g * IB + b * CB + c * LB;
          uint32_t q0w[F::kLaneWords], q1w[F::kLaneWords];
          F::lds_lane(cr, q0w);
          F::lds_lane(cr + 8 * IB, q1w);
          uint32_t f0[4], f1[4];
          F::decode_lane(q0w, f0);
          F::decode_lane(q1w, f1);
          const float s0 = ue8m0_to_f32(st[L.codes + g * nbI + b]);
          const float s1 = ue8m0_to_f32(st[L.codes + (g + 8) * nbI + b]);
          // token g's block b, this lane's eight elements, as f16 (zeros for a
          // column past the pass's tokens)
          const uint4 hv = tg ? *reinterpret_cast<const uint4*>(hb + 64 * b)
                              : make_uint4(0u, 0u, 0u, 0u);
          uint32_t xb[4];
          const float fx = quad_block_f16(hv, xb);
          const float fa = __shfl_sync(kFull, fx, 8 * c);       // column 2c (quad 2c)
          const float fb = __shfl_sync(kFull, fx, 8 * c + 4);   // column 2c+1
          float cb[4] = {0.f, 0.f, 0.f, 0.f};
          mma_16816(cb, f0[0], f1[0], f0[1], f1[1], xb[0], xb[1]);
          mma_16816(cb, f0[2], f1[2], f0[3], f1[3], xb[2], xb[3]);
          acc[0] = fmaf(cb[0], s0 * fa, acc[0]);
          acc[1] = fmaf(cb[1], s0 * fb, acc[1]);
          acc[2] = fmaf(cb[2], s1 * fa, acc[2]);
          acc[3] = fmaf(cb[3], s1 * fb, acc[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      // rows g, g+8 x columns 2c, 2c+1 of the item, times the columns' routing
      // weights, into this warp's accumulator (distinct addresses per lane)
      if (!dead) {
        if (2 * c < nt) {
          const int t = tl[2 * c];
          yw[t * kDmRows + g] += tw[2 * c] * acc[0];
          yw[t * kDmRows + g + 8] += tw[2 * c] * acc[2];
        }
        if (2 * c + 1 < nt) {
          const int t = tl[2 * c + 1];
          yw[t * kDmRows + g] += tw[2 * c + 1] * acc[1];
          yw[t * kDmRows + g + 8] += tw[2 * c + 1] * acc[3];
        }
      }
    }
    named_sync(1, ncons);   // every item of the tile is in the accumulators
    for (int i = threadIdx.x; i < p.T * kDmRows; i += ncons) {
      float v = 0.f;
      for (int w = 0; w < kDmConsumers; ++w) v += yacc[w * p.T * kDmRows + i];
      const int t = i / kDmRows, n = i - t * kDmRows;
      p.y[(size_t)t * H + r0 + n] = dead ? (uint16_t)0 : f32_to_bf16_rn(v);
    }
    named_sync(1, ncons);   // the accumulators read before the next tile clears them
  }
}

}  // namespace moe
