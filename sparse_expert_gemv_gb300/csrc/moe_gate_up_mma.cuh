// Gate/up for several tokens: TMA-streamed weight tiles, products on the
// tensor cores' warp-level MMA.
//
// The warp-decode post (cursor.com/blog/warp-decode, "How the two kernels
// work") streams each routed expert's gate and up rows once per step and
// applies them to every token routed to the expert. With several tokens per
// expert each weight meets several activation vectors, and the FP32 path
// (one warp per neuron, moe_gate_up_3d_batched_xs) spends more instructions
// per product on decoding, activation loads and FMAs than the SM can issue:
// at 32 tokens it is bound by instruction issue, not by HBM, and at 8 by the
// few loads each warp keeps in flight. This kernel changes both:
//
//   * The stream. One producer warp per CTA walks the CTA's work items, each
//     a tile of 16 consecutive neurons of one unique expert together with up
//     to eight of that expert's tokens, and streams the tile's gate and up
//     rows (and scales) through a ring of shared-memory slots with TMA tensor
//     copies, K-chunk by K-chunk (512 code bytes of each row per slot). The
//     items are split over the CTAs in equal shares, so every CTA streams the
//     same number of bytes.
//   * The products. All 16 consumer warps work on the same slot, each on its
//     own 32-element K blocks, with mma.sync m16n8k16 (f16 operands, FP32
//     accumulation): A = the tile's 16 decoded weight rows (M), B = the
//     tokens' staged activations (N = 8), two MMAs per block. At the end of
//     an item the warps' partial sums meet in shared memory and are added in
//     a fixed order (no atomics: results are reproducible bit for bit).
//
// Exactness is that of the FP32 path: E4M3 and E2M1 codes are exact in f16,
// x is staged as f16 blocks scaled by a power of two (moe_f16blocks.cuh), the
// MMA's f16 products are exact and accumulate in FP32, and each block's sum
// is multiplied by the block's weight scale and activation factor in FP32.
//
// Fragment layout. In m16n8k16 lane (g, c) = (lane / 4, lane % 4) supplies K
// positions 2c, 2c+1, 2c+8, 2c+9 of A rows g and g+8 and of B column g. A dot
// product does not depend on the order of K, so positions are mapped to
// actual K such that a lane's four positions of the first MMA of a block are
// the block's elements 8c .. 8c+3 and those of the second MMA 8c+4 .. 8c+7:
// each lane reads eight consecutive codes of each of its rows per block and
// 16 consecutive bytes of its token's staged activations.
#pragma once

#include <cuda.h>

#include "moe_kernels.cuh"

namespace moe {

constexpr int kGuConsumers = 16;                         // consumer warps
constexpr int kGuThreads = (kGuConsumers + 1) * 32;      // + one producer warp
constexpr int kGuRows = 16;                              // neurons per tile (the MMA's M)
constexpr int kGuTokens = 8;                             // tokens per item (the MMA's N)
constexpr int kGuRowBytes = 512;                         // code bytes of a row per ring slot

// Bytes between two tokens' staged x rows: H f16 values plus 16, so that the
// 16-byte loads of eight tokens mostly fall in different bank groups.
__host__ __device__ constexpr int mma_xrow(int H) { return H * 2 + 16; }

struct GateUpTmaParams {
  // W_gateup codes as a 3D uint32 tensor [E*2I][RB/512][128] with boxes of
  // 16 rows x 512 bytes, and its scales as a 2D uint32 tensor [E*2I][H/128]
  // with boxes of 16 rows x KC/32 scale bytes (RB = code bytes per row)
  CUtensorMap tm_codes;
  CUtensorMap tm_scales;
  const uint16_t* x;      // [T, H] bf16
  const int32_t* ids;     // [T, k]
  uint16_t* h;            // [T, k, I] bf16
  uint32_t* err;
  int T, k, E, H, I;
  int KC;                 // weights of a row per slot: 512 code bytes (512 MXFP8, 1024 MXFP4)
  int SG;                 // ring slots
};

// A ring slot is a code slot (1024-byte aligned: gate codes, then up codes)
// and a scale slot (gate scales [16][KC/32], then up scales). Each matrix's
// codes are four [16][128] pieces (row bytes 0-127, 128-255, ...) written by
// TMA with the 128-byte swizzle: 16-byte chunk j of row r sits at chunk
// j ^ (r % 8), so the 16 rows' chunks a warp reads at once fall in
// different banks.
struct GuSlot {
  int codes, us, scales;   // code slot bytes, up scales' offset, scale slot bytes
  __host__ __device__ explicit GuSlot(int KC)
      : codes(2 * kGuRows * kGuRowBytes),
        us(round128(kGuRows * (KC >> 5))),
        scales(2 * round128(kGuRows * (KC >> 5))) {}
};

// Address of byte o (< 512) of row r of a matrix's codes in a slot.
__device__ __forceinline__ const uint8_t* gu_code(const uint8_t* m, int r, int o) {
  return m + (o >> 7) * (kGuRows * 128) + r * 128 + ((((o >> 4) & 7) ^ (r & 7)) << 4) + (o & 15);
}

// Shared-memory map (byte offsets, 128-byte aligned): the ring, x as f16
// rows, their block factors, two buffers for the warps' partial sums, the
// mbarriers, the warps' schedule words, each consumer warp's token list of
// its current item, and the prefix counts of items.
struct GuTmaSmem {
  int slot, sslot, sc, xs, xf, red, bars, words, tl, pref, total;
  // offsets from the first 1024-byte boundary of the dynamic shared memory
  // (total includes the up to 1024 bytes before it); the code slots first,
  // then the scale slots
  __host__ __device__ GuTmaSmem(int SG, int KC, int T, int H, int nU_max) {
    const GuSlot gs(KC);
    slot = gs.codes;
    sslot = gs.scales;
    int o = SG * slot;
    sc = o;
    o += SG * sslot;
    xs = o;
    o += round128(T * mma_xrow(H));
    xf = o;
    o += round128(T * (H >> 5) * 4);
    red = o;
    o += 2 * kGuConsumers * 32 * 8 * 4;
    bars = o;
    o += round128(2 * SG * 8);
    words = o;
    o += (kGuConsumers + 1) * 32 * 4;
    tl = o;
    o += kGuConsumers * 2 * kGuTokens * 4;
    pref = o;
    o += round128((nU_max + 1) * 4);
    total = o + 1024;
  }
};

// d += A x B for one m16n8k16 tile (f16 A and B, FP32 accumulators).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The CTA's work items in order: unique expert u (ascending), its tiles of
// 16 neurons, and for each tile the expert's tokens in passes of eight.
// pref[u] = sum of passes of the unique experts below u, so the items of
// expert u are tpe * pref[u] .. tpe * pref[u+1] - 1. Producer and consumers
// run the same walk.
struct GuItems {
  int x, hi, tpe, u, pu, np, tile, pass;
  const int* pref;
  __device__ __forceinline__ void begin(const int* pref_, int nU, int tpe_) {
    pref = pref_;
    tpe = tpe_;
    const long long total = (long long)tpe * pref[nU];
    x = (int)(total * blockIdx.x / gridDim.x);
    hi = (int)(total * (blockIdx.x + 1) / gridDim.x);
    if (x >= hi) return;
    // the expert holding item x: the last u with tpe * pref[u] <= x
    int lo_u = 0, hi_u = nU - 1;
    while (lo_u < hi_u) {
      const int mid = (lo_u + hi_u + 1) >> 1;
      if ((long long)tpe * pref[mid] <= x) lo_u = mid; else hi_u = mid - 1;
    }
    u = lo_u;
    pu = pref[u];
    np = pref[u + 1] - pu;
    const int r = x - tpe * pu;
    tile = r / np;
    pass = r - tile * np;
  }
  __device__ __forceinline__ bool valid() const { return x < hi; }
  __device__ __forceinline__ void next() {
    ++x;
    if (++pass < np) return;
    pass = 0;
    if (++tile < tpe) return;
    tile = 0;
    if (x >= hi) return;
    ++u;
    pu = pref[u];
    np = pref[u + 1] - pu;
  }
};

template <int KMAX, class F>
__global__ void __launch_bounds__(kGuThreads, 1) moe_gate_up_tma(const __grid_constant__ GateUpTmaParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the swizzled TMA copies need 1024-byte aligned destinations
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  constexpr int CB = F::kBlockBytes, LB = F::kLaneBytes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int H = p.H, I = p.I, nb = H >> 5, KC = p.KC, SG = p.SG;
  const int nbk = KC >> 5;                  // blocks per slot (16 MXFP8, 32 MXFP4)
  const int nkc = H / KC;                   // slots per tile
  const int xrow = mma_xrow(H);
  const int nU_max = min(p.E, p.T * p.k);
  const GuTmaSmem L(SG, KC, p.T, H, nU_max);
  const GuSlot sl(KC);
  uint8_t* sring = smem + L.sc;
  uint8_t* ring = smem;
  uint8_t* xs = smem + L.xs;
  float* xf = reinterpret_cast<float*>(smem + L.xf);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + SG;
  uint32_t* sm_words = reinterpret_cast<uint32_t*>(smem + L.words);
  int* pref = reinterpret_cast<int*>(smem + L.pref);
  const int ncons = kGuConsumers * 32;
  if (warp == kGuConsumers && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_codes) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_scales) : "memory");
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < SG; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGuConsumers);
    }
    mbar_init_fence();
  }
  pdl_wait();      // x and topk_ids come from upstream work
  pdl_trigger();   // the down kernel may start fetching its weights
  WarpSchedule<KMAX> s;
  s.load(p.ids, p.T, p.k);
  if (warp < kGuConsumers) {
    // x -> f16 rows (blocks in natural chunk order) while the ids are in flight
#pragma unroll 1
    for (int idx = threadIdx.x; idx < p.T * nb; idx += ncons) {
      const int t = idx / nb, b = idx - t * nb;
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * H) + 4 * b;
      const uint4 v[4] = {__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3)};
      xf[idx] = stage_block_f16(v, xs + (size_t)t * xrow + 64 * b, 0);
    }
  }
  s.finish(p.E, sm_words + warp * 32, p.err);
  const int nU = s.n_unique;
  // passes of each unique expert (its tokens in groups of eight)
#pragma unroll 1
  for (int u = warp; u < nU; u += kGuConsumers + 1) {
    const int e = s.expert(u);
    const int n = __popc(__ballot_sync(kFull, s.jmask(e) != 0u));
    if (lane == 0) pref[u + 1] = (n + kGuTokens - 1) / kGuTokens;
  }
  // A slot with an out-of-range id gets no item; its h slice is defined as zero.
  if (warp < kGuConsumers && __any_sync(kFull, s.badmask != 0u)) {
    for (int t = blockIdx.x * kGuConsumers + warp; t < p.T; t += gridDim.x * kGuConsumers) {
      const uint32_t bm = __shfl_sync(kFull, s.badmask, t);
      for (uint32_t m = bm; m; m &= m - 1) {
        uint16_t* row = p.h + ((size_t)t * p.k + (__ffs(m) - 1)) * I;
        for (int i = lane; i < I; i += 32) row[i] = 0;
      }
    }
  }
  __syncthreads();   // x staged, pass counts written
  if (warp == 0) {
    // inclusive scan of the pass counts into item prefixes
    int carry = 0;
    if (lane == 0) pref[0] = 0;
    for (int base = 1; base <= nU; base += 32) {
      const int i = base + lane;
      int v = i <= nU ? pref[i] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int w = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += w;
      }
      if (i <= nU) pref[i] = carry + v;
      carry += __shfl_sync(kFull, v, 31);
    }
  }
  __syncthreads();   // prefixes written
  const int tpe = I / kGuRows;

  if (warp == kGuConsumers) {
    // ------------------------------------------------------------ producer
    GuItems it;
    it.begin(pref, nU, tpe);
    RingPos rg(SG);
    int gi = 0;
    bool ok = true;
#pragma unroll 1
    for (; ok && it.valid(); it.next()) {
      const int e = s.expert(it.u);   // warp-collective
      const int row = e * 2 * I + it.tile * kGuRows;
#pragma unroll 1
      for (int kc = 0; kc < nkc; ++kc, rg.next(), ++gi) {
        if (lane == 0 && gi >= SG) ok = mbar_wait(&empty[rg.slot], rg.phase ^ 1u, p.err);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* dst = ring + (size_t)rg.slot * L.slot;
          uint64_t* bar = &full[rg.slot];
          mbar_expect_tx(bar, 2u * kGuRows * kGuRowBytes + 2u * kGuRows * (KC >> 5));
          for (int q = 0; q < kGuRowBytes / 128; ++q) {
            tma_load_3d(dst + q * kGuRows * 128, &p.tm_codes, 0, kc * (kGuRowBytes / 128) + q, row,
                        bar);
            tma_load_3d(dst + kGuRows * kGuRowBytes + q * kGuRows * 128, &p.tm_codes, 0,
                        kc * (kGuRowBytes / 128) + q, row + I, bar);
          }
          uint8_t* sdst = sring + (size_t)rg.slot * L.sslot;
          tma_load_2d(sdst, &p.tm_scales, kc * (KC >> 7), row, bar);
          tma_load_2d(sdst + sl.us, &p.tm_scales, kc * (KC >> 7), row + I, bar);
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
  // a warp whose bounded wait gave up stops waiting and computing but still
  // reaches every arrival and named barrier, so no other warp can hang on it
  bool dead = false;
  GuItems it;
  it.begin(pref, nU, tpe);
  RingPos rg(SG);
  int rb = 0;   // partial-sum buffer of this item
  const int bpw = nbk / kGuConsumers;   // blocks per warp per slot (1 MXFP8, 2 MXFP4)
  // this warp's token list of the current item: token ids, then their slot masks
  int* tl = reinterpret_cast<int*>(smem + L.tl) + warp * 2 * kGuTokens;
  uint32_t* tj = reinterpret_cast<uint32_t*>(tl + kGuTokens);
  int cur_u = -1;
  uint32_t jm = 0, tokens = 0;
#pragma unroll 1
  for (; it.valid(); it.next()) {
    if (it.u != cur_u) {
      // the expert changes: its tokens (lane t: token t's slots of the expert)
      cur_u = it.u;
      jm = s.jmask(s.expert(it.u));
      tokens = __ballot_sync(kFull, jm != 0u);
    }
    const int base = kGuTokens * it.pass;
    const int nt = min(kGuTokens, __popc(tokens) - base);
    {
      // tokens base .. base+nt-1 of the expert, in ascending order
      const int rank = __popc(tokens & ((1u << lane) - 1u)) - base;
      __syncwarp();
      if (jm != 0u && rank >= 0 && rank < kGuTokens) {
        tl[rank] = lane;
        tj[rank] = jm;
      }
      __syncwarp();
    }
    const int tok_g = g < nt ? tl[g] : -1;
    const int tok_a = 2 * c < nt ? tl[2 * c] : -1;
    const int tok_b = 2 * c + 1 < nt ? tl[2 * c + 1] : -1;
    const uint8_t* xrow_g = xs + (size_t)(tok_g < 0 ? 0 : tok_g) * xrow + 16 * c;
    const float* xf_a = xf + (size_t)(tok_a < 0 ? 0 : tok_a) * nb;
    const float* xf_b = xf + (size_t)(tok_b < 0 ? 0 : tok_b) * nb;
    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int kc = 0; kc < nkc; ++kc, rg.next()) {
      if (!dead) dead = !mbar_wait(&full[rg.slot], rg.phase, p.err);
      // the MMAs below need the whole warp: a wait that ran out on any lane
      // stops them on every lane
      dead = __any_sync(kFull, dead);
      if (!dead) {
        const uint8_t* st = ring + (size_t)rg.slot * L.slot;
        const uint8_t* ss = sring + (size_t)rg.slot * L.sslot;
#pragma unroll
        for (int bi = 0; bi < 2; ++bi) {
          if (bi < bpw) {
            const int blk = warp * bpw + bi;          // block within the slot
            const int b = kc * nbk + blk;             // block of the row
            const int o = blk * CB + c * LB;             // byte of the slot's row chunk
            const uint8_t* upm = st + kGuRows * kGuRowBytes;
            uint32_t q[4][F::kLaneWords];
            F::lds_lane(gu_code(st, g, o), q[0]);
            F::lds_lane(gu_code(st, g + 8, o), q[1]);
            F::lds_lane(gu_code(upm, g, o), q[2]);
            F::lds_lane(gu_code(upm, g + 8, o), q[3]);
            uint32_t fg0[4], fg1[4], fu0[4], fu1[4];
            F::decode_lane(q[0], fg0);
            F::decode_lane(q[1], fg1);
            F::decode_lane(q[2], fu0);
            F::decode_lane(q[3], fu1);
            const float s_g0 = ue8m0_to_f32(ss[g * nbk + blk]);
            const float s_g1 = ue8m0_to_f32(ss[(g + 8) * nbk + blk]);
            const float s_u0 = ue8m0_to_f32(ss[sl.us + g * nbk + blk]);
            const float s_u1 = ue8m0_to_f32(ss[sl.us + (g + 8) * nbk + blk]);
            const uint4 xb = tok_g >= 0 ? *reinterpret_cast<const uint4*>(xrow_g + 64 * b)
                                        : make_uint4(0u, 0u, 0u, 0u);
            const float fa = tok_a >= 0 ? xf_a[b] : 0.f;
            const float fb = tok_b >= 0 ? xf_b[b] : 0.f;
            float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(cg, fg0[0], fg1[0], fg0[1], fg1[1], xb.x, xb.y);
            mma_16816(cg, fg0[2], fg1[2], fg0[3], fg1[3], xb.z, xb.w);
            mma_16816(cu, fu0[0], fu1[0], fu0[1], fu1[1], xb.x, xb.y);
            mma_16816(cu, fu0[2], fu1[2], fu0[3], fu1[3], xb.z, xb.w);
            ag[0] = fmaf(cg[0], s_g0 * fa, ag[0]);
            ag[1] = fmaf(cg[1], s_g0 * fb, ag[1]);
            ag[2] = fmaf(cg[2], s_g1 * fa, ag[2]);
            ag[3] = fmaf(cg[3], s_g1 * fb, ag[3]);
            au[0] = fmaf(cu[0], s_u0 * fa, au[0]);
            au[1] = fmaf(cu[1], s_u0 * fb, au[1]);
            au[2] = fmaf(cu[2], s_u1 * fa, au[2]);
            au[3] = fmaf(cu[3], s_u1 * fb, au[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[rg.slot]);
    }
    // the 16 warps' partial sums of this item, added in a fixed order: warp n
    // takes neuron n of the tile, lane quad q token column q, and the four
    // lanes of the quad a quarter of the warps each, then a two-step tree
    float* red = reinterpret_cast<float*>(smem + L.red) + rb * (kGuConsumers * 32 * 8);
    reinterpret_cast<float4*>(red)[(warp * 32 + lane) * 2] = make_float4(ag[0], ag[1], ag[2], ag[3]);
    reinterpret_cast<float4*>(red)[(warp * 32 + lane) * 2 + 1] = make_float4(au[0], au[1], au[2], au[3]);
    named_sync(1, ncons);
    {
      const int n = warp, col = lane >> 2, w0 = 4 * (lane & 3);
      // output (n, col) sits in fragment lane (n % 8) * 4 + col / 2, element
      // 2 * (n / 8) + col % 2
      const int L2 = (n & 7) * 4 + (col >> 1), r = 2 * (n >> 3) + (col & 1);
      float gs = 0.f, us = 0.f;
      if (col < nt) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          gs += red[((w0 + w) * 32 + L2) * 8 + r];
          us += red[((w0 + w) * 32 + L2) * 8 + 4 + r];
        }
      }
      gs += __shfl_xor_sync(kFull, gs, 1);
      us += __shfl_xor_sync(kFull, us, 1);
      gs += __shfl_xor_sync(kFull, gs, 2);
      us += __shfl_xor_sync(kFull, us, 2);
      if ((lane & 3) == 0 && col < nt && !dead) {
        const uint16_t hb = f32_to_bf16_rn((gs / (1.0f + expf(-gs))) * us);
        const int tok = tl[col];
        for (uint32_t m = tj[col]; m; m &= m - 1)
          p.h[((size_t)tok * p.k + (__ffs(m) - 1)) * I + it.tile * kGuRows + n] = hb;
      }
    }
    rb ^= 1;
  }
}

}  // namespace moe
