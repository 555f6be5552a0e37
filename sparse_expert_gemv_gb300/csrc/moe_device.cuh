// Device building blocks shared by the decode-layer kernels: PTX wrappers for
// streaming loads, MXFP8 element/scale decode, bf16 handling, warp reductions,
// programmatic-dependent-launch controls and the per-warp expert dedup
// schedule.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kDeviceBadId = 0x1u;

// ---------------------------------------------------------------------------
// loads
// ---------------------------------------------------------------------------

// 32 bytes of a weight row that is read once per step: no L1 allocation, and
// an L2 eviction-first hint so the stream does not push activations out.
__device__ __forceinline__ void ld_weights32(const uint8_t* p, uint32_t (&r)[8]) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "l"(p));
}

// 16 bytes of activations that many warps re-read: keep them in L1 and L2.
__device__ __forceinline__ uint4 ld_act16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::evict_last.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16 bytes of a weight row read once per step (the 32 codes of one MXFP4
// block): no L1 allocation (the L2 eviction-priority form of the load exists
// for 256-bit accesses only).
__device__ __forceinline__ void ld_weights16(const uint8_t* p, uint32_t (&r)[4]) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "l"(p));
}

__device__ __forceinline__ uint32_t ld_scale(const uint8_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// TMA bulk copies, mbarriers, named barriers
// ---------------------------------------------------------------------------

constexpr uint32_t kDeviceTimeout = 0x2u;   // a bounded wait gave up
constexpr uint32_t kWaitLimit = 1u << 22;   // polls before a spin wait gives up
// mbarrier waits suspend for up to kWaitSuspendNs per poll (waking as soon as
// the phase completes) and give up after kMbarPolls polls (about a second)
constexpr uint32_t kWaitSuspendNs = 20000;
constexpr uint32_t kMbarPolls = 1u << 16;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also announces `bytes` of copies completing on the barrier.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

// Wait for the phase with the given parity to complete. Gives up after
// kMbarPolls polls, sets kDeviceTimeout in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, uint32_t* err) {
#pragma unroll 1
  for (uint32_t it = 0; it < kMbarPolls; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(b)), "r"(parity), "r"(kWaitSuspendNs)
        : "memory");
    if (done) return true;
  }
  atomicOr(err, kDeviceTimeout);
  return false;
}

// Whether the phase with the given parity has completed, without waiting.
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(b)), "r"(parity)
      : "memory");
  return done != 0;
}

// Global -> shared bulk copy completing on an mbarrier. Source and
// destination 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 2D tile of a tensor map (x = innermost coordinate in elements, y = row) ->
// shared memory, completing on an mbarrier. x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// 3D tile of a tensor map (x innermost, in elements) -> shared memory,
// completing on an mbarrier. x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// 4D tile of a tensor map (x innermost, in elements) -> shared memory,
// completing on an mbarrier. x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}

__host__ __device__ constexpr int round128(int v) { return (v + 127) / 128 * 128; }

// Position in a ring of n shared-memory slots: slot index and the parity of
// its current fill.
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

// Barrier over `nthreads` threads (whole warps) of the CTA on named barrier `id`.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// MXFP8 decode
// ---------------------------------------------------------------------------

// Four E4M3 codes (byte n = element n) to FP32. The hardware conversion to
// f16 is exact for every finite E4M3 value (f16 covers 2^-14..65504 with 10
// mantissa bits; E4M3 spans 2^-9..448 with 3), and f16 -> f32 is exact.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t q, float& f0, float& f1, float& f2,
                                              float& f3) {
  uint32_t lo, hi;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(q));
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(f0), "=f"(f1)
      : "r"(lo));
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(f2), "=f"(f3)
      : "r"(hi));
}

// UE8M0 scale code s -> 2^(s-127) as FP32, built from its bit pattern:
// exponent field s for s >= 1, the subnormal 2^-127 for s = 0, NaN for 0xFF.
__device__ __forceinline__ float ue8m0_to_f32(uint32_t s) {
  uint32_t bits = s << 23;
  bits = (s == 0u) ? 0x00400000u : bits;
  bits = (s == 255u) ? 0x7fc00000u : bits;
  return __uint_as_float(bits);
}

// ---------------------------------------------------------------------------
// bf16
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// FP32 -> bf16 bits, round to nearest even (NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// ---------------------------------------------------------------------------
// warp reductions (the butterfly of the warp-decode post, "How the two
// kernels work": shfl.sync.bfly, no shared memory, no barrier)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// The tokens of one pass over a unit's rows: the lowest NT set bits of the
// unit's token mask (grp holds them only for groups kept as a mask). Groups of up to four keep the token indices in
// registers; larger groups keep only the mask and walk it where a token is
// needed, leaving their NT registers to the accumulators.
template <int NT>
struct TokenGroup {
  static constexpr bool kMask = NT > 4;
  int tok[kMask ? 1 : NT];
  uint32_t grp;   // the group's tokens
  int nt;         // how many (<= NT)
  // Takes the group from `tokens` (removing it there).
  __device__ __forceinline__ void take(uint32_t& tokens) {
    if constexpr (kMask) {
      uint32_t rest = tokens;
#pragma unroll
      for (int n = 0; n < NT; ++n) rest &= rest - 1;   // drop the lowest NT
      grp = tokens ^ rest;
      nt = __popc(grp);
      tokens = rest;
    } else {
      grp = 0u;
      nt = 0;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        tok[n] = tokens ? __ffs(tokens) - 1 : 0;
        if (tokens) {
          tokens &= tokens - 1;
          ++nt;
        }
      }
    }
  }
  // Token n of the group, for n = 0, 1, ... in order; `walk` starts at grp.
  __device__ __forceinline__ int token(int n, uint32_t& walk) const {
    if constexpr (kMask) {
      const int t = __ffs(walk) - 1;
      walk &= walk - 1;
      return t;
    } else {
      return tok[n];
    }
  }
};

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------

// Block until the grids this one depends on have completed and their memory
// is visible. A no-op when the kernel was not launched as a dependent.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next grid on the stream to start launching its blocks.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------------------
// Per-warp expert dedup schedule for up to 32 tokens.
//
// Lane t holds token t's k expert ids. The set of routed experts is a bitmap
// over E (word w held by lane w, E <= 1024); its popcount prefix numbers the
// unique experts in ascending id order. For a given expert, each lane reports
// which of its slots j route there (jmask), and a ballot gives the tokens.
// Everything lives in registers plus per-warp shared memory (32 bitmap words,
// and with IdStore::kShared the packed ids), so each warp builds it alone
// with no block barrier.
// ---------------------------------------------------------------------------

// Where a schedule keeps its lanes' ids after finish(): in registers, or in
// a [(KMAX + 1) / 2][32]-word table of the warp's shared memory (lane-minor,
// so a lane's reads are conflict-free), which gives the registers back to
// kernels that hold many tokens' accumulators through their main loop.
enum class IdStore { kRegisters, kShared };

// Shared-memory bytes of one warp's id table for IdStore::kShared.
__host__ __device__ constexpr int schedule_id_bytes(int kmax) { return (kmax + 1) / 2 * 32 * 4; }

// The several-token warp kernels keep a token's ids in registers when there
// are at most eight slots and the kernel holds at most two tokens'
// accumulators at a time, else in shared memory (where registers would
// spill).
template <int NT, int KMAX>
constexpr IdStore kWarpIdStore = KMAX > 8 || NT > 2 ? IdStore::kShared : IdStore::kRegisters;

template <int KMAX, IdStore S = IdStore::kRegisters>
struct WarpSchedule {
  static constexpr int kIdWords = (KMAX + 1) / 2;
  static constexpr bool kShared = S == IdStore::kShared;
  int id[KMAX];      // this lane's token's ids as loaded (dead after finish())
  // the same after finish(), two to a word (slot j in bits 16 (j & 1) of word
  // j / 2; 0xFFFF: slot unused or invalid): in registers, or in word j / 2 of
  // this lane's column of the warp's shared table
  uint32_t idp[kShared ? 1 : kIdWords];
  uint32_t* idcol;   // IdStore::kShared: this lane's column (stride 32 words)
  uint32_t badmask;  // slots j of this lane's token whose id is outside [0, E)
  uint32_t word;     // routed-expert bitmap word `lane`
  int excl;          // unique experts in words below `lane`
  int n_unique;

  // sm_ids: the warp's id table (schedule_id_bytes(KMAX) bytes) with
  // IdStore::kShared, unused otherwise.
  __device__ __forceinline__ void build(const int32_t* __restrict__ ids, int T, int k, int E,
                                        uint32_t* sm_words, uint32_t* err,
                                        uint32_t* sm_ids = nullptr) {
    load(ids, T, k);
    finish(E, sm_words, err, sm_ids);
  }

  // The two halves of build(): load() only issues the id loads, so that
  // independent work can run while they are in flight before finish().
  __device__ __forceinline__ void load(const int32_t* __restrict__ ids, int T, int k) {
    const int lane = threadIdx.x & 31;
    badmask = 0u;   // slots in use until finish()
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      id[j] = -1;
      if (lane < T && j < k) {
        id[j] = __ldg(ids + lane * k + j);
        badmask |= 1u << j;
      }
    }
  }
  __device__ __forceinline__ void finish(int E, uint32_t* sm_words, uint32_t* err,
                                         uint32_t* sm_ids = nullptr) {
    const int lane = threadIdx.x & 31;
    const uint32_t used = badmask;
    badmask = 0u;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (((used >> j) & 1u) && (id[j] < 0 || id[j] >= E)) {
        badmask |= 1u << j;
        id[j] = -1;
      }
    }
    if (badmask) atomicOr(err, kDeviceBadId);
    if constexpr (kShared) idcol = sm_ids + lane;
#pragma unroll
    for (int w = 0; w < kIdWords; ++w) {
      const uint32_t lo = id[2 * w] < 0 ? 0xFFFFu : (uint32_t)id[2 * w];
      const uint32_t hi = 2 * w + 1 >= KMAX || id[2 * w + 1] < 0 ? 0xFFFFu : (uint32_t)id[2 * w + 1];
      if constexpr (kShared)
        idcol[32 * w] = lo | (hi << 16);
      else
        idp[w] = lo | (hi << 16);
    }
    sm_words[lane] = 0u;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (id[j] >= 0) atomicOr(&sm_words[id[j] >> 5], 1u << (id[j] & 31));
    __syncwarp();
    word = sm_words[lane];
    __syncwarp();
    const int cnt = __popc(word);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    excl = incl - cnt;
    n_unique = __shfl_sync(kFull, incl, 31);
  }

  // Expert id of the u-th unique expert (ascending), 0 <= u < n_unique.
  __device__ __forceinline__ int expert(int u) const {
    const int lane = threadIdx.x & 31;
    const unsigned owner = __ballot_sync(kFull, u >= excl && u < excl + __popc(word));
    const int L = __ffs(owner) - 1;
    const uint32_t w = __shfl_sync(kFull, word, L);
    const int n = u - __shfl_sync(kFull, excl, L);     // n-th set bit of w (0-based)
    const bool mine = ((w >> lane) & 1u) && (__popc(w & ((1u << lane) - 1u)) == n);
    return L * 32 + (__ffs(__ballot_sync(kFull, mine)) - 1);
  }

  // Expert id of the u-th unique expert where u differs per lane (every lane
  // takes part; a lane with u >= n_unique gets an unspecified value): the
  // owner word is the first whose inclusive prefix count exceeds u, found by
  // a five-step binary search over the lanes' prefix counts.
  __device__ __forceinline__ int expert_per_lane(int u) const {
    const int incl = excl + __popc(word);
    int L = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
      if (__shfl_sync(kFull, incl, L + step - 1) <= u) L += step;
    const uint32_t w = __shfl_sync(kFull, word, L & 31);
    const int n = u - __shfl_sync(kFull, excl, L & 31);
    return (L & 31) * 32 + (int)__fns(w, 0, n + 1);
  }

  // Slot j's id after finish() (-1: unused or invalid).
  __device__ __forceinline__ int idj(int j) const {
    uint32_t wd;
    if constexpr (kShared)
      wd = idcol[32 * (j >> 1)];
    else
      wd = idp[j >> 1];
    const uint32_t v = (wd >> (16 * (j & 1))) & 0xFFFFu;
    return v == 0xFFFFu ? -1 : (int)v;
  }

  // Bits j of this lane's token whose id equals e.
  __device__ __forceinline__ uint32_t jmask(int e) const {
    uint32_t m = 0;
    if constexpr (kShared) {
      // one shared load per two slots (e is a valid id, never 0xFFFF)
#pragma unroll
      for (int w = 0; w < kIdWords; ++w) {
        const uint32_t wd = idcol[32 * w];
        m |= ((wd & 0xFFFFu) == (uint32_t)e ? 1u : 0u) << (2 * w);
        if (2 * w + 1 < KMAX) m |= ((wd >> 16) == (uint32_t)e ? 1u : 0u) << (2 * w + 1);
      }
    } else {
#pragma unroll
      for (int j = 0; j < KMAX; ++j) m |= (idj(j) == e ? 1u : 0u) << j;
    }
    return m;
  }
};

}  // namespace moe
