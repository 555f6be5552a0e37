// Host side of the C ABI declared in include/moe_decode.h: argument checks,
// handle lifetime, launch configuration and the programmatic-dependent-launch
// chaining of the two projection kernels.
#include "moe_decode.h"
#include "moe_decode_timeline.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <new>

#include "moe_down_mma.cuh"
#include "moe_down_tma.cuh"
#include "moe_gate_up_mma.cuh"
#include "moe_kernels.cuh"
#include "moe_layer_fused.cuh"
#include "moe_tc.cuh"

namespace {

constexpr int kMaxE = 1024;  // the schedule's expert bitmap is 32 words
constexpr int kMaxK = 32;    // a token's slots are bits of one 32-bit mask
constexpr int kVersion = 100;
// h[t] (k*I FP32 values) is staged in shared memory by the down kernel
constexpr size_t kMaxDownSmem = 200 * 1024;

}  // namespace

struct moe_decode {
  moe_decode_config_t cfg;
  const uint8_t* wgu;
  const uint8_t* sgu;
  const uint8_t* wd;
  const uint8_t* sd;
  int device;
  int num_sms;
  int gate_up_ctas_per_sm;
  size_t down_smem;
  size_t smem_per_block;          // opt-in shared-memory maximum of one CTA
  bool fused_ok;                  // the single-token fused kernel can run here
  bool host_direct;               // the device reads pageable host memory coherently
  CUtensorMap tm_codes;           // W_gateup codes / scales and W_down codes / scales
  CUtensorMap tm_scales;          // as tensors for its TMA copies
  CUtensorMap tm_dcodes;
  CUtensorMap tm_dscales;
  bool gu_tma_ok;                 // the several-token TMA gate/up kernel can run here
  CUtensorMap tm_gu_codes;        // its W_gateup codes / scales tensor maps
  CUtensorMap tm_gu_scales;
  bool dn_tma_ok;                 // the several-token TMA down kernel can run here
  CUtensorMap tm_dn_codes;        // its W_down codes / scales tensor maps
  CUtensorMap tm_dn_scales;
  uint32_t* d_err;                // device error word (4 bytes) ...
  unsigned long long* d_bar;      // ... then, 8 and 16 bytes on, the fused kernel's launch
                                  // and grid-barrier counters
  // completion of the handle's latest enqueued call (recorded outside stream
  // capture), which moe_decode_get_error waits for, and a private
  // non-blocking stream for reading and clearing the error word
  cudaEvent_t done_ev;
  bool done_recorded;
  cudaStream_t aux;
  // the expert-centric tensor-core path (moe_tc.cuh): whether it can run
  // (shape, alignment, and every weight decoding to a normal bf16), which
  // path calls take (MOE_PATH_*), its workspace for min(max_T, 256) * k
  // pairs, its tensor maps (W_gateup codes and scales, W_down codes, xg, hg),
  // ring depths and shared-memory sizes
  bool tc_ok;
  bool tc_f16_gu;                 // its gate/up weights decode exactly to f16 (moe_tc_gate_up<F, true>)
  int path;
  void* tc_mem;
  moe::TcWork tcw;
  CUtensorMap tm_tc_gu;
  CUtensorMap tm_tc_gus;
  CUtensorMap tm_tc_dn;
  CUtensorMap tm_tc_x;
  CUtensorMap tm_tc_h;
  int tc_R_gu, tc_R_dn;
  size_t tc_smem_gu, tc_smem_dn;
  // staging buffers of moe_decode_forward_host (max_T tokens)
  uint16_t* d_x;
  int32_t* d_ids;
  float* d_w;
  uint16_t* d_h;
  uint16_t* d_y;
};

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The device address of a page-locked host buffer mapped into the device's
// address space, or null (pageable memory, or a device pointer).
const void* mapped_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

template <typename Kernel, typename... Args>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                   Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

bool use_pdl(const moe_decode* m) { return (m->cfg.flags & MOE_FLAG_NO_PDL) == 0; }

// The handle's weight format: MXFP4 (E2M1 codes, two to a byte) or MXFP8.
bool is_fp4(const moe_decode* m) { return (m->cfg.flags & MOE_FLAG_MXFP4) != 0; }
int code_bytes_per_block(const moe_decode* m) { return is_fp4(m) ? 16 : 32; }

constexpr uint32_t kKnownFlags =
    MOE_FLAG_NO_PDL | MOE_FLAG_HOST_COPY | MOE_FLAG_MXFP4 | MOE_FLAG_WARP_MMA;

// The KMAX instance of the warp kernels for this handle's k (8 or 32).
int kmax_of(const moe_decode* m) { return m->cfg.k <= 8 ? 8 : 32; }

// Whether several-token warp-decode calls may take the warp-level MMA kernels.
bool warp_mma(const moe_decode* m) { return (m->cfg.flags & MOE_FLAG_WARP_MMA) != 0; }

// ---- gate/up ---------------------------------------------------------------

// Fewest tokens of a gate/up launch that takes moe_gate_up_tma.
constexpr int kGuTmaMinTokens = 16;

// Weights of a row per ring slot of moe_gate_up_tma: 512 code bytes.
int gu_tma_kc(const moe_decode* m) { return moe::kGuRowBytes * 32 / code_bytes_per_block(m); }

// Ring slots of moe_gate_up_tma for T tokens: as many as fit beside the
// staged x (at most 16), 0 when fewer than two fit.
int gu_tma_slots(const moe_decode* m, int T, size_t& smem) {
  const moe_decode_config_t& c = m->cfg;
  const int KC = gu_tma_kc(m), nU_max = std::min(c.E, T * c.k);
  auto bytes = [&](int SG) { return (size_t)moe::GuTmaSmem(SG, KC, T, c.H, nU_max).total; };
  if (bytes(2) > m->smem_per_block) return 0;
  int SG = 2;
  while (SG < 16 && bytes(SG + 1) <= m->smem_per_block) ++SG;
  smem = bytes(SG);
  return SG;
}

template <int KMAX, class F>
cudaError_t launch_gate_up_tma(const moe_decode* m, const moe::GateUpParams& p, int SG,
                               size_t smem, cudaStream_t s) {
  moe::GateUpTmaParams q;
  q.tm_codes = m->tm_gu_codes;
  q.tm_scales = m->tm_gu_scales;
  q.x = p.x;
  q.ids = p.ids;
  q.h = p.h;
  q.err = p.err;
  q.T = p.T;
  q.k = p.k;
  q.E = p.E;
  q.H = p.H;
  q.I = p.I;
  q.KC = gu_tma_kc(m);
  q.SG = SG;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(m->num_sms);
  cfg.blockDim = dim3(moe::kGuThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = use_pdl(m) ? attr : nullptr;
  cfg.numAttrs = use_pdl(m) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, moe::moe_gate_up_tma<KMAX, F>, q);
}

// The gate/up kernel of a launch of T tokens (at most 32), with its ring
// slots and shared memory where it has a ring.
enum class GuKind { kTma, kXs, kL1 };
GuKind gate_up_kind(const moe_decode* m, int T, int& SG, size_t& smem) {
  // with MOE_FLAG_WARP_MMA, sixteen or more tokens whose x fits in shared
  // memory beside a weight ring: tiles streamed by TMA, products on the
  // warp-level MMA (one CTA per SM). It pays when an expert serves many
  // tokens; where each serves one or two (uniform routing) the FP32 kernel
  // below issues fewer instructions per weight byte (T = 16: 132 against
  // 240 us a layer).
  if (warp_mma(m) && T >= kGuTmaMinTokens && m->gu_tma_ok) {
    SG = gu_tma_slots(m, T, smem);
    if (SG >= 2) return GuKind::kTma;
  }
  // several tokens whose x fits in shared memory: staged once per CTA as f16
  // blocks (one 16-warp CTA per SM)
  smem = moe::gate_up_xs_smem(T, m->cfg.H, kmax_of(m));
  if (T >= 2 && smem <= m->smem_per_block) return GuKind::kXs;
  return GuKind::kL1;
}

template <int NT, int KMAX, class F, int D>
cudaError_t launch_gate_up_xs(const moe_decode* m, const moe::GateUpParams& p, size_t xs,
                              cudaStream_t s) {
  const long long units_max = (long long)std::min(p.E, p.T * p.k) * p.I;
  const long long ctas_needed = (units_max + moe::kXsWarps - 1) / moe::kXsWarps;
  const int grid = (int)std::max(1LL, std::min(ctas_needed, (long long)m->num_sms));
  return launch(moe::moe_gate_up_3d_batched_xs<NT, KMAX, F, D>, dim3(grid), dim3(moe::kXsThreads),
                xs, s, use_pdl(m), p);
}

template <int NT, int KMAX, class F>
cudaError_t launch_gate_up_t(const moe_decode* m, const moe::GateUpParams& p, cudaStream_t s) {
  int SG = 0;
  size_t smem = 0;
  const GuKind kind = gate_up_kind(m, p.T, SG, smem);
  if (kind == GuKind::kTma) return launch_gate_up_tma<KMAX, F>(m, p, SG, smem, s);
  if (kind == GuKind::kXs) {
    // at most one token per expert on average (T*k <= E): token groups of two
    // and two weight blocks per lane in flight (the registers of larger
    // token groups go to the stream instead)
    if ((long long)p.T * p.k <= p.E) return launch_gate_up_xs<2, KMAX, F, 2>(m, p, smem, s);
    return launch_gate_up_xs<NT, KMAX, F, 1>(m, p, smem, s);
  }
  const long long units_max = (long long)std::min(p.E, p.T * p.k) * p.I;
  const long long ctas_needed = (units_max + moe::kWarps - 1) / moe::kWarps;
  const long long cap = (long long)m->num_sms * m->gate_up_ctas_per_sm;
  const int grid = (int)std::max(1LL, std::min(ctas_needed, cap));
  return launch(moe::moe_gate_up_3d_batched<NT, KMAX, F>, dim3(grid), dim3(moe::kThreads), 0, s,
                use_pdl(m), p);
}

template <int KMAX, class F>
cudaError_t launch_gate_up_k(const moe_decode* m, const moe::GateUpParams& p, cudaStream_t s) {
  if (p.T <= 1) return launch_gate_up_t<1, KMAX, F>(m, p, s);
  if (p.T <= 2) return launch_gate_up_t<2, KMAX, F>(m, p, s);
  if (p.T <= 4) return launch_gate_up_t<4, KMAX, F>(m, p, s);
  return launch_gate_up_t<8, KMAX, F>(m, p, s);
}

template <class F>
cudaError_t launch_gate_up_f(const moe_decode* m, const moe::GateUpParams& p, cudaStream_t s) {
  if (p.k <= 8) return launch_gate_up_k<8, F>(m, p, s);
  return launch_gate_up_k<32, F>(m, p, s);
}

cudaError_t launch_gate_up(const moe_decode* m, const moe::GateUpParams& p, cudaStream_t s) {
  return is_fp4(m) ? launch_gate_up_f<moe::Mxfp4>(m, p, s) : launch_gate_up_f<moe::Mxfp8>(m, p, s);
}

// ---- down ------------------------------------------------------------------

// Weight blocks a lane keeps in flight in moe_down_3d_batched: eight MXFP4
// blocks (16 code bytes each) or six MXFP8 ones (32 bytes each), as many as
// fit its 128 registers without spilling (a warp's 32 x 6 blocks still cover
// the k I / 32 = 192 blocks of a 768-wide expert at k = 8 in one round).
template <class F>
constexpr int kDownQ = F::kBlockBytes == 16 ? 8 : 6;

// Ring slots of moe_down_tma: as many as fit beside h (at most 16), 0 when
// fewer than two fit.
int dn_tma_slots(const moe_decode* m, size_t& smem) {
  const moe_decode_config_t& c = m->cfg;
  const int IB = c.I / 32 * code_bytes_per_block(m);
  auto bytes = [&](int SG) { return (size_t)moe::DnTmaSmem(SG, c.I, IB, c.k).total; };
  if (bytes(2) > m->smem_per_block) return 0;
  int SG = 2;
  while (SG < 16 && bytes(SG + 1) <= m->smem_per_block) ++SG;
  smem = bytes(SG);
  return SG;
}

template <class F>
cudaError_t launch_down_tma(const moe_decode* m, const moe::DownParams& p, int SG, size_t smem,
                            cudaStream_t s) {
  moe::DownTmaParams q;
  q.tm_codes = m->tm_dn_codes;
  q.tm_scales = m->tm_dn_scales;
  q.h = p.h;
  q.ids = p.ids;
  q.w = p.w;
  q.y = p.y;
  q.err = p.err;
  q.T = p.T;
  q.k = p.k;
  q.E = p.E;
  q.H = p.H;
  q.I = p.I;
  q.SG = SG;
  const long long items = (long long)p.T * (p.H / moe::kDnRows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<long long>(items, m->num_sms));
  cfg.blockDim = dim3(moe::kDnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = use_pdl(m) ? attr : nullptr;
  cfg.numAttrs = use_pdl(m) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, moe::moe_down_tma<F>, q);
}

// Fewest ring slots (and so reducing warps) with which moe_down_mma is used.
constexpr int kDnMmaMinSlots = 6;

int dn_tma_slots(const moe_decode* m, size_t& smem);
int dn_mma_slots(const moe_decode* m, int T, size_t& smem);

// The down kernel of a launch of T tokens (at most 32), with its ring slots
// and shared memory where it has a ring.
enum class DnKind { kMma, kTma, kWarp };
DnKind down_kind(const moe_decode* m, int T, int& SG, size_t& smem) {
  // sixteen or more tokens with rows of at most 1 KB of codes: each unique
  // expert's row tiles streamed once, products on the warp-level MMA (with
  // fewer tokens an expert rarely serves more than one or two, and the
  // token-by-token kernel keeps more of the stream in flight; a warp per ring
  // slot: with few slots too few warps would reduce)
  if (warp_mma(m) && T >= kGuTmaMinTokens && m->dn_tma_ok &&
      m->cfg.I / 32 * code_bytes_per_block(m) <= 1024) {
    SG = dn_mma_slots(m, T, smem);
    if (SG >= kDnMmaMinSlots) return DnKind::kMma;
  }
  // several tokens otherwise: the TMA-streamed kernel, token by token
  if (T >= 2 && m->dn_tma_ok) {
    SG = dn_tma_slots(m, smem);
    if (SG >= 2) return DnKind::kTma;
  }
  smem = moe::down_xs_smem(m->cfg.k, m->cfg.I);
  return DnKind::kWarp;
}

// Ring slots of moe_down_mma for T tokens: as many as fit, at most one per
// consumer warp; 0 when fewer than two fit.
int dn_mma_slots(const moe_decode* m, int T, size_t& smem) {
  const moe_decode_config_t& c = m->cfg;
  const int IB = c.I / 32 * code_bytes_per_block(m), nU_max = std::min(c.E, T * c.k);
  auto bytes = [&](int SG) { return (size_t)moe::DmSmem(SG, c.I, IB, T, nU_max, kmax_of(m)).total; };
  if (bytes(2) > m->smem_per_block) return 0;
  int SG = 2;
  while (SG < moe::kDmConsumers && bytes(SG + 1) <= m->smem_per_block) ++SG;
  smem = bytes(SG);
  return SG;
}

template <int KMAX, class F>
cudaError_t launch_down_mma(const moe_decode* m, const moe::DownParams& p, int SG, size_t smem,
                            cudaStream_t s) {
  moe::DownMmaParams q;
  q.tm_codes = m->tm_dn_codes;
  q.tm_scales = m->tm_dn_scales;
  q.h = p.h;
  q.ids = p.ids;
  q.w = p.w;
  q.y = p.y;
  q.err = p.err;
  q.T = p.T;
  q.k = p.k;
  q.E = p.E;
  q.H = p.H;
  q.I = p.I;
  q.SG = SG;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(p.H / moe::kDmRows, m->num_sms));
  cfg.blockDim = dim3(moe::kDmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = use_pdl(m) ? attr : nullptr;
  cfg.numAttrs = use_pdl(m) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, moe::moe_down_mma<KMAX, F>, q);
}

template <class F>
cudaError_t launch_down_mma_k(const moe_decode* m, const moe::DownParams& p, int SG, size_t smem,
                              cudaStream_t s) {
  return p.k <= 8 ? launch_down_mma<8, F>(m, p, SG, smem, s) : launch_down_mma<32, F>(m, p, SG, smem, s);
}

cudaError_t launch_down(const moe_decode* m, const moe::DownParams& p, cudaStream_t s) {
  int SG = 0;
  size_t smem = 0;
  const DnKind kind = down_kind(m, p.T, SG, smem);
  if (kind == DnKind::kMma)
    return is_fp4(m) ? launch_down_mma_k<moe::Mxfp4>(m, p, SG, smem, s)
                     : launch_down_mma_k<moe::Mxfp8>(m, p, SG, smem, s);
  if (kind == DnKind::kTma)
    return is_fp4(m) ? launch_down_tma<moe::Mxfp4>(m, p, SG, smem, s)
                     : launch_down_tma<moe::Mxfp8>(m, p, SG, smem, s);
  const dim3 grid(p.H / moe::kWarps, p.T), block(moe::kThreads);
  if (is_fp4(m))
    return launch(moe::moe_down_3d_batched<kDownQ<moe::Mxfp4>, moe::Mxfp4>, grid, block, smem, s, use_pdl(m), p);
  return launch(moe::moe_down_3d_batched<kDownQ<moe::Mxfp8>, moe::Mxfp8>, grid, block, smem, s, use_pdl(m), p);
}

// The down kernels' shared-memory limit: one value for every handle, the
// library's maximum (the TMA kernels': the device's opt-in maximum).
cudaError_t set_down_attributes() {
  cudaError_t e = cudaSuccess;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return cudaErrorUnknown;
  for (const void* f : {(const void*)moe::moe_down_tma<moe::Mxfp8>,
                        (const void*)moe::moe_down_tma<moe::Mxfp4>,
                        (const void*)moe::moe_down_mma<8, moe::Mxfp8>,
                        (const void*)moe::moe_down_mma<32, moe::Mxfp8>,
                        (const void*)moe::moe_down_mma<8, moe::Mxfp4>,
                        (const void*)moe::moe_down_mma<32, moe::Mxfp4>})
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  for (const void* f : {(const void*)moe::moe_down_3d_batched<kDownQ<moe::Mxfp8>, moe::Mxfp8>,
                        (const void*)moe::moe_down_3d_batched<kDownQ<moe::Mxfp4>, moe::Mxfp4>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDownSmem);
  return e;
}

// ---- single-token fused layer ----------------------------------------------

int gcd_int(int a, int b) { return b ? gcd_int(b, a % b) : a; }

// Ring geometry of moe_layer_fused_t1 for this handle's shape; false when the
// shape or the pointers do not suit it (the two-kernel path is used instead).
// The ring carries the CTA's gate/up tiles and then its down row groups, as
// many slots as fit beside the staged x and h.
bool plan_fused(const moe_decode* m, moe::FusedParams& fp, size_t& smem) {
  const moe_decode_config_t& c = m->cfg;
  if (!m->fused_ok || c.H % 512 || c.I % 128 || !aligned(m->sgu, 16) || !aligned(m->sd, 16))
    return false;
  const int CB = code_bytes_per_block(m);
  const int nbI = c.I / 32, IB = nbI * CB;
  const int RG = 16 / gcd_int(16, nbI);
  if (c.H % RG) return false;
  const int rows_cta = (c.H / RG + m->num_sms - 1) / m->num_sms * RG;
  constexpr int kMaxSlots = 16;
  // a stage's K-chunk, by its code bytes per row: the first of these that H
  // allows and the ring holds (1 KB stages put the first tiles to work sooner
  // than 2 KB ones and free ring slots for the down rows earlier)
  for (const int KB : {1024, 2048, 512}) {
    const int KC = KB / CB * 32;
    if (c.H % KC) continue;
    const int slot_g = moe::GuStageLayout(KB, KC).end;    // a multiple of 128
    // down row chunks of RC rows, as many as the consumers cover and a slot holds
    int RC = std::min(rows_cta, moe::kFusedConsumers / RG * RG);
    while (RC >= RG && moe::round128(RC * (IB + nbI)) > slot_g) RC -= RG;
    if (RC < RG) continue;
    const int slot_d = moe::round128(RC * (IB + nbI));
    const int SR = slot_g / slot_d;
    auto bytes = [&](int SG) { return (size_t)moe::FusedSmem(SG, slot_g, c.H, c.I, c.k).total; };
    if (bytes(2) > m->smem_per_block) continue;
    int SG = 2;
    while (SG < kMaxSlots && bytes(SG + 1) <= m->smem_per_block) ++SG;
    // every group of a row chunk is resident at once
    if ((c.k + SR - 1) / SR > SG) continue;
    smem = bytes(SG);
    fp.KC = KC;
    fp.kin = std::min(256, KB / 4);
    fp.SG = SG;
    fp.slot_g = slot_g;
    fp.SR = SR;
    fp.slot_d = slot_d;
    fp.RG = RG;
    fp.RC = RC;
    fp.nkc = c.H / KC;
    fp.kdiv = KB / (4 * fp.kin);
    fp.nrg = c.H / RG;
    return true;
  }
  return false;
}

// cuTensorMapEncodeTiled from the driver, looked up once (no link to libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A [rows, cols] uint32 matrix with a row pitch of `pitch` bytes, read in
// boxes of box_rows x box_cols.
bool encode_u32_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch,
                   uint32_t box_cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [rows, n1, n0] uint32 tensor (n0 innermost, rows `pitch` bytes apart),
// read in boxes of box_rows x b1 x n0, written to shared memory as is or
// with the 128-byte swizzle (then n0 * 4 must be 128).
bool encode_u32_3d(CUtensorMap* tm, const void* base, uint64_t n0, uint64_t n1, uint64_t rows,
                   uint64_t pitch, uint32_t b1, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {n0, n1, rows};
  cuuint64_t strides[2] = {n0 * 4, pitch};
  cuuint32_t box[3] = {(cuuint32_t)n0, b1, box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [n3, n2, n1, n0] uint32 tensor (n0 innermost, dense), read in boxes of
// 1 x b2 x n1 x n0.
bool encode_u32_4d(CUtensorMap* tm, const void* base, uint64_t n0, uint64_t n1, uint64_t n2,
                   uint64_t n3, uint32_t b2) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[4] = {n0, n1, n2, n3};
  cuuint64_t strides[3] = {n0 * 4, n0 * n1 * 4, n0 * n1 * n2 * 4};
  cuuint32_t box[4] = {(cuuint32_t)n0, (cuuint32_t)n1, b2, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The fused kernel's tensor maps (code bytes per row: RB = H*CB/32 for
// W_gateup, IB = I*CB/32 for W_down, KB = KC*CB/32 per K-chunk, CB the code
// bytes of a 32-element block). W_gateup codes as [E*2I][RB/(4*kin)][kin]
// uint32 with boxes of kFusedNeurons rows x KB bytes, its scales as
// [E*2I][H/128] uint32 with boxes of kFusedNeurons rows x KC/32 scale bytes;
// W_down codes as [E][H][IB/(4*kin_d)][kin_d] uint32 with boxes of RC rows of
// one expert, its scales as [E][H*I/128] uint32 with boxes of RC rows.
bool encode_fused_maps(moe_decode* m, int KC, int RC) {
  const moe_decode_config_t& c = m->cfg;
  const int CB = code_bytes_per_block(m);
  const int RB = c.H / 32 * CB, IB = c.I / 32 * CB, KB = KC / 32 * CB;
  const uint64_t rows = (uint64_t)c.E * 2 * c.I;
  const int kin = std::min(256, KB / 4);
  const int kin_d = std::min(256, IB / 4);
  return encode_u32_3d(&m->tm_codes, m->wgu, kin, RB / (4 * kin), rows, RB, KB / (4 * kin),
                       moe::kFusedNeurons) &&
         encode_u32_2d(&m->tm_scales, m->sgu, c.H / 128, rows, c.H / 32, KC / 128,
                       moe::kFusedNeurons) &&
         encode_u32_4d(&m->tm_dcodes, m->wd, kin_d, IB / (4 * kin_d), c.H, c.E, RC) &&
         encode_u32_2d(&m->tm_dscales, m->sd, (uint64_t)c.H * c.I / 128, c.E,
                       (uint64_t)c.H * c.I / 32, RC * c.I / 128, 1);
}

// The several-token gate/up kernel's tensor maps: W_gateup codes as
// [E*2I][RB/128][32] uint32 with boxes of 16 rows x 128 bytes written with
// the 128-byte swizzle, its scales as [E*2I][H/128] uint32 with boxes of 16
// rows x KC/32 scale bytes. False when the shape or the scale pointer does
// not suit them.
bool gu_tma_shape_ok(const moe_decode* m) {
  return m->cfg.H % gu_tma_kc(m) == 0 && aligned(m->sgu, 16);
}

bool encode_gu_tma_maps(moe_decode* m) {
  const moe_decode_config_t& c = m->cfg;
  const int KC = gu_tma_kc(m);
  if (!gu_tma_shape_ok(m)) return false;
  const int RB = c.H / 32 * code_bytes_per_block(m);
  const uint64_t rows = (uint64_t)c.E * 2 * c.I;
  return encode_u32_3d(&m->tm_gu_codes, m->wgu, 32, RB / 128, rows, RB, 1, moe::kGuRows,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_u32_2d(&m->tm_gu_scales, m->sgu, c.H / 128, rows, c.H / 32, KC / 128,
                       moe::kGuRows);
}

// The several-token down kernel's tensor maps: W_down codes as
// [E][H][IB/(4*kin)][kin] uint32 with boxes of one expert's 16 rows, its
// scales as [E][H*I/128] uint32 with boxes of 16 rows' scale bytes. False
// when the shape or the pointers do not suit them (I a multiple of 128 and at
// most 2048, scale array 16-byte aligned).
bool dn_tma_shape_ok(const moe_decode* m) {
  return m->cfg.I % 128 == 0 && m->cfg.I <= 2048 && aligned(m->sd, 16);
}

bool encode_dn_tma_maps(moe_decode* m) {
  const moe_decode_config_t& c = m->cfg;
  if (!dn_tma_shape_ok(m)) return false;
  const int IB = c.I / 32 * code_bytes_per_block(m);
  const int kin = std::min(256, IB / 4);
  return encode_u32_4d(&m->tm_dn_codes, m->wd, kin, IB / (4 * kin), c.H, c.E, moe::kDnRows) &&
         encode_u32_2d(&m->tm_dn_scales, m->sd, (uint64_t)c.H * c.I / 128, c.E,
                       (uint64_t)c.H * c.I / 32, moe::kDnRows * c.I / 128, 1);
}

cudaError_t set_fused_attributes(size_t smem) {
  cudaError_t e = cudaSuccess;
  for (const void* f : {(const void*)moe::moe_layer_fused_t1<8, moe::Mxfp8>,
                        (const void*)moe::moe_layer_fused_t1<32, moe::Mxfp8>,
                        (const void*)moe::moe_layer_fused_t1<8, moe::Mxfp4>,
                        (const void*)moe::moe_layer_fused_t1<32, moe::Mxfp4>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return e;
}

// One persistent CTA per SM; cooperative so that every CTA is resident for
// the grid barrier between the two phases.
cudaError_t launch_fused(const moe_decode* m, const moe::FusedParams& fp, size_t smem,
                         cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(m->num_sms);
  cfg.blockDim = dim3(moe::kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl(m) ? 2 : 1;
  if (is_fp4(m)) {
    if (fp.k <= 8) return cudaLaunchKernelEx(&cfg, moe::moe_layer_fused_t1<8, moe::Mxfp4>, fp);
    return cudaLaunchKernelEx(&cfg, moe::moe_layer_fused_t1<32, moe::Mxfp4>, fp);
  }
  if (fp.k <= 8) return cudaLaunchKernelEx(&cfg, moe::moe_layer_fused_t1<8, moe::Mxfp8>, fp);
  return cudaLaunchKernelEx(&cfg, moe::moe_layer_fused_t1<32, moe::Mxfp8>, fp);
}

// Device limits shared by handles and the allocation-free call: SM count,
// gate/up occupancy, shared memory, and whether the fused kernel fits one CTA
// per SM (it then runs as a cooperative launch of num_sms CTAs).
// The shared-memory limit of the gate/up kernels that stage x: the device's
// opt-in maximum.
template <class F>
cudaError_t set_xs_attributes_f(size_t smem) {
  cudaError_t e = cudaSuccess;
  for (const void* f : {(const void*)moe::moe_gate_up_3d_batched_xs<1, 8, F, 1>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<2, 8, F, 1>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<4, 8, F, 1>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<8, 8, F, 1>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<2, 8, F, 2>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<1, 32, F, 1>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<2, 32, F, 1>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<4, 32, F, 1>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<8, 32, F, 1>,
                        (const void*)moe::moe_gate_up_3d_batched_xs<2, 32, F, 2>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return e;
}

cudaError_t set_xs_attributes(size_t smem) {
  cudaError_t e = set_xs_attributes_f<moe::Mxfp8>(smem);
  if (e == cudaSuccess) e = set_xs_attributes_f<moe::Mxfp4>(smem);
  for (const void* f : {(const void*)moe::moe_gate_up_tma<8, moe::Mxfp8>,
                        (const void*)moe::moe_gate_up_tma<32, moe::Mxfp8>,
                        (const void*)moe::moe_gate_up_tma<8, moe::Mxfp4>,
                        (const void*)moe::moe_gate_up_tma<32, moe::Mxfp4>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return e;
}

bool query_fused(moe_decode* m) {
  int v_blk = 0, coop = 0;
  if (cudaDeviceGetAttribute(&v_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, m->device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, m->device) != cudaSuccess)
    return false;
  m->smem_per_block = (size_t)v_blk;
  if (set_xs_attributes(m->smem_per_block) != cudaSuccess) return false;
  m->fused_ok = false;
  if (!coop || set_fused_attributes(m->smem_per_block) != cudaSuccess) return true;
  moe::FusedParams fp = {};
  size_t smem = 0;
  m->fused_ok = true;
  if (!plan_fused(m, fp, smem)) {
    m->fused_ok = false;
    return true;
  }
  int occ = 0;
  const void* fk = is_fp4(m) ? (const void*)moe::moe_layer_fused_t1<8, moe::Mxfp4>
                             : (const void*)moe::moe_layer_fused_t1<8, moe::Mxfp8>;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fk, moe::kFusedThreads, smem) !=
      cudaSuccess)
    return false;
  m->fused_ok = occ >= 1 && encode_fused_maps(m, fp.KC, fp.RC);
  return true;
}

moe_status_t fused_layer(moe_decode* m, const uint16_t* x, const int32_t* ids, const float* w,
                         uint16_t* h, uint16_t* y, cudaStream_t s,
                         unsigned long long* stamps = nullptr) {
  moe::FusedParams fp = {};
  size_t smem = 0;
  plan_fused(m, fp, smem);
  const moe_decode_config_t& c = m->cfg;
  fp.x = x;
  fp.ids = ids;
  fp.w = w;
  fp.wgu = m->wgu;
  fp.sgu = m->sgu;
  fp.wd = m->wd;
  fp.sd = m->sd;
  fp.h = h;
  fp.y = y;
  fp.err = m->d_err;
  fp.launch_ctr = m->d_bar;
  fp.bar_ctr = m->d_bar + 1;
  fp.stamps = stamps;
  fp.tm_codes = m->tm_codes;
  fp.tm_scales = m->tm_scales;
  fp.tm_dcodes = m->tm_dcodes;
  fp.tm_dscales = m->tm_dscales;
  fp.k = c.k;
  fp.E = c.E;
  fp.H = c.H;
  fp.I = c.I;
  return launch_fused(m, fp, smem, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---- expert-centric tensor-core path (moe_tc.cuh) --------------------------

// MOE_PATH_AUTO takes the tensor-core path from kTcAutoMinTokens tokens when
// they route at least 1.5 slots per expert on average (2 T k >= 3 E).
// Measured on one GB300 (E = 128, k = 8, H = 2048, I = 768, MXFP8, us a
// layer, FP32 warp kernels / tensor-core path): uniform routing T = 16
// 132 / 154, T = 24 192 / 178, T = 32 238 / 194; Zipf-skewed routing
// T = 16 128 / 82, T = 24 178 / 88, T = 32 232 / 91. E = 256 at T = 16 (one
// slot per two experts): 916 / 1412.
constexpr int kTcAutoMinTokens = 16;

// Shapes the path's kernels cover: whole 128-row tiles of I and H, gate/up
// scale chunks of 512 elements, 16-byte aligned scale arrays, and TMA row
// coordinates (E * 2I, E * H) that fit an int.
bool tc_shape_ok(const moe_decode* m) {
  const moe_decode_config_t& c = m->cfg;
  return c.H % 512 == 0 && c.I % 128 == 0 && aligned(m->sgu, 16) && aligned(m->sd, 16) &&
         (int64_t)c.E * 2 * c.I < (int64_t)INT32_MAX && (int64_t)c.E * c.H < (int64_t)INT32_MAX;
}

int tc_pairs(const moe_decode* m) { return std::min(m->cfg.max_T, moe::kTcMaxTokens) * m->cfg.k; }

// Whether every weight decodes to a normal bf16 (scale codes in range, no
// E4M3 NaN code): one pass over both projections' codes and scales. False
// with ok = false when a CUDA call failed.
bool tc_weights_exact(moe_decode* m, bool& ok) {
  const moe_decode_config_t& c = m->cfg;
  const int CB = code_bytes_per_block(m);
  uint32_t* d = nullptr;
  // gate/up's scale range and NaN flag, then down's
  const uint32_t init[8] = {0xFFFFFFFFu, 0u, 0u, 0u, 0xFFFFFFFFu, 0u, 0u, 0u};
  uint32_t h[8] = {};
  const size_t gu_scales = (size_t)c.E * 2 * c.I * (c.H / 32);
  const size_t dn_scales = (size_t)c.E * c.H * (c.I / 32);
  const size_t gu_codes = gu_scales * CB, dn_codes = dn_scales * CB;
  const dim3 grid(m->num_sms * 4), block(256);
  (void)cudaGetLastError();   // a launch error below must be this pass's own
  ok = cudaMalloc(&d, 32) == cudaSuccess &&
       cudaMemcpy(d, init, 32, cudaMemcpyHostToDevice) == cudaSuccess;
  if (ok) {
    moe::moe_tc_scan<<<grid, block>>>(reinterpret_cast<const uint4*>(m->wgu), gu_codes / 16,
                                      reinterpret_cast<const uint4*>(m->sgu), gu_scales / 16,
                                      is_fp4(m) ? 0 : 1, d);
    moe::moe_tc_scan<<<grid, block>>>(reinterpret_cast<const uint4*>(m->wd), dn_codes / 16,
                                      reinterpret_cast<const uint4*>(m->sd), dn_scales / 16,
                                      is_fp4(m) ? 0 : 1, d + 4);
    ok = cudaGetLastError() == cudaSuccess &&
         cudaMemcpy(h, d, 32, cudaMemcpyDeviceToHost) == cudaSuccess;
  }
  if (d) cudaFree(d);
  const uint32_t lo = is_fp4(m) ? moe::kTcScaleMinFp4 : moe::kTcScaleMinFp8;
  const uint32_t f16_hi = is_fp4(m) ? moe::kTcF16ScaleMaxFp4 : moe::kTcF16ScaleMaxFp8;
  // the gate/up weights in f16 when their scale codes allow it
  m->tc_f16_gu = ok && h[0] >= (uint32_t)moe::kTcF16ScaleMin && h[1] <= f16_hi && h[2] == 0u;
  return ok && std::min(h[0], h[4]) >= lo && std::max(h[1], h[5]) <= (uint32_t)moe::kTcScaleMax &&
         h[2] == 0u && h[6] == 0u;
}

// A [rows, cols] tensor of `dtype` (elem bytes each, rows `pitch` bytes
// apart) read in boxes of box_rows x box_cols.
bool encode_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base, uint64_t cols,
               uint64_t rows, uint64_t pitch, uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, dtype, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Deepest weight-code ring (at most 32 slots) whose kernel fits the
// shared-memory limit, with the 1024-byte alignment slack; 0 when none does.
int tc_ring(const moe_decode* m, bool down, size_t& smem) {
  const int RB = is_fp4(m) ? moe::TcFp4::kStageRowBytes : moe::TcFp8::kStageRowBytes;
  for (int R = 32; R >= 4; --R) {
    const moe::TcSmem L(down, RB, R, m->cfg.I);
    if ((size_t)L.total + 1024 <= m->smem_per_block) {
      smem = (size_t)L.total + 1024;
      return R;
    }
  }
  return 0;
}

template <class F>
cudaError_t set_tc_attributes(size_t gu, size_t dn, size_t prep) {
  cudaError_t e = cudaFuncSetAttribute(moe::moe_tc_gate_up<F, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gu);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(moe::moe_tc_gate_up<F, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gu);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(moe::moe_tc_down<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(moe::moe_tc_prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)prep);
  return e;
}

// Sets m->tc_ok when the path can run for this handle: allocates its
// workspace and encodes its tensor maps. False only when a CUDA call failed.
bool tc_setup(moe_decode* m) {
  m->tc_ok = false;
  const moe_decode_config_t& c = m->cfg;
  if (c.max_T < 1 || !tc_shape_ok(m)) return true;
  bool ok = true;
  if (!tc_weights_exact(m, ok)) return ok;
  size_t smem_gu = 0, smem_dn = 0;
  m->tc_R_gu = tc_ring(m, false, smem_gu);
  m->tc_R_dn = tc_ring(m, true, smem_dn);
  const int Pw = tc_pairs(m);
  // moe_tc_prep's dynamic shared memory for a full group (its 16 static
  // bytes come on top)
  const size_t smem_prep = moe::tc_prep_smem(Pw, c.E);
  if (m->tc_R_gu == 0 || m->tc_R_dn == 0 || smem_prep + 256 > m->smem_per_block) return true;
  m->tc_smem_gu = smem_gu;
  m->tc_smem_dn = smem_dn;
  // workspace: schedule ints, then xg, hg and yp (256-byte aligned)
  const int maxC = std::min(c.E, Pw) + Pw / moe::kTcCols + 1;
  auto up256 = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t ints = up256((size_t)(4 + 3 * maxC + 2 * Pw) * 4);
  const size_t xg = up256((size_t)Pw * c.H * 2), hg = up256((size_t)Pw * c.I * 2);
  const size_t yp = up256((size_t)Pw * c.H * 4), xi = up256((size_t)Pw * 4);
  if (cudaMalloc(&m->tc_mem, ints + xg + hg + yp + xi) != cudaSuccess ||
      cudaMemset(m->tc_mem, 0, ints + xg + hg + yp + xi) != cudaSuccess)
    return false;
  uint8_t* b = static_cast<uint8_t*>(m->tc_mem);
  int* iw = reinterpret_cast<int*>(b);
  m->tcw.hdr = iw;
  m->tcw.chunk_e = iw + 4;
  m->tcw.chunk_p0 = m->tcw.chunk_e + maxC;
  m->tcw.chunk_n = m->tcw.chunk_p0 + maxC;
  m->tcw.pair_slot = m->tcw.chunk_n + maxC;
  m->tcw.slot_pair = m->tcw.pair_slot + Pw;
  m->tcw.xg = reinterpret_cast<uint16_t*>(b + ints);
  m->tcw.hg = reinterpret_cast<uint16_t*>(b + ints + xg);
  m->tcw.yp = reinterpret_cast<float*>(b + ints + xg + hg);
  m->tcw.xinv = reinterpret_cast<float*>(b + ints + xg + hg + yp);
  const int CB = code_bytes_per_block(m);
  const int RB = is_fp4(m) ? moe::TcFp4::kStageRowBytes : moe::TcFp8::kStageRowBytes;
  const CUtensorMapSwizzle sw = is_fp4(m) ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
  const uint64_t gu_rows = (uint64_t)c.E * 2 * c.I, dn_rows = (uint64_t)c.E * c.H;
  const uint64_t gu_rb = (uint64_t)c.H / 32 * CB, dn_rb = (uint64_t)c.I / 32 * CB;
  const bool maps =
      encode_2d(&m->tm_tc_gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, m->wgu, gu_rb, gu_rows, gu_rb, RB,
                moe::kTcRows, sw) &&
      encode_2d(&m->tm_tc_gus, CU_TENSOR_MAP_DATA_TYPE_UINT8, m->sgu, c.H / 32, gu_rows,
                c.H / 32, 16, moe::kTcRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
      encode_2d(&m->tm_tc_dn, CU_TENSOR_MAP_DATA_TYPE_UINT8, m->wd, dn_rb, dn_rows, dn_rb, RB,
                moe::kTcRows, sw) &&
      encode_2d(&m->tm_tc_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, m->tcw.xg, c.H, Pw, (uint64_t)c.H * 2,
                moe::kTcK, moe::kTcBBox, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_2d(&m->tm_tc_h, CU_TENSOR_MAP_DATA_TYPE_UINT16, m->tcw.hg, c.I, Pw, (uint64_t)c.I * 2,
                moe::kTcK, moe::kTcBBox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!maps) return true;
  const cudaError_t e =
      is_fp4(m) ? set_tc_attributes<moe::TcFp4>(smem_gu, smem_dn, smem_prep)
                : set_tc_attributes<moe::TcFp8>(smem_gu, smem_dn, smem_prep);
  if (e != cudaSuccess) return false;
  m->tc_ok = true;
  return true;
}

// Whether a call with T tokens takes the tensor-core path.
bool use_tc(const moe_decode* m, int T) {
  if (!m->tc_ok || m->path == MOE_PATH_WARP) return false;
  return m->path == MOE_PATH_TENSOR ||
         (T >= kTcAutoMinTokens && 2 * T * m->cfg.k >= 3 * m->cfg.E);
}

template <class F>
moe_status_t tc_layer_f(moe_decode* m, int T, const uint16_t* x, const int32_t* ids,
                        const float* w, uint16_t* h, uint16_t* y, cudaStream_t s) {
  const moe_decode_config_t& c = m->cfg;
  const bool pdl = use_pdl(m);
  for (int t0 = 0; t0 < T; t0 += moe::kTcMaxTokens) {
    const int Tg = std::min(moe::kTcMaxTokens, T - t0);
    const int P = Tg * c.k;
    moe::TcPrepParams pp = {};
    pp.x = x + (size_t)t0 * c.H;
    pp.ids = ids + (size_t)t0 * c.k;
    pp.h = h + (size_t)t0 * c.k * c.I;
    pp.err = m->d_err;
    pp.w = m->tcw;
    pp.T = Tg;
    pp.k = c.k;
    pp.E = c.E;
    pp.H = c.H;
    pp.I = c.I;
    pp.f16 = m->tc_f16_gu ? 1 : 0;
    moe::TcParams gp = {};
    gp.tm_w = m->tm_tc_gu;
    gp.tm_s = m->tm_tc_gus;
    gp.tm_b = m->tm_tc_x;
    gp.sd = m->sd;
    gp.h = pp.h;
    gp.err = m->d_err;
    gp.w = m->tcw;
    gp.E = c.E;
    gp.H = c.H;
    gp.I = c.I;
    gp.R = m->tc_R_gu;
    moe::TcParams dp = gp;
    dp.tm_w = m->tm_tc_dn;
    dp.tm_b = m->tm_tc_h;
    dp.R = m->tc_R_dn;
    moe::TcCombineParams cp = {};
    cp.tw = w + (size_t)t0 * c.k;
    cp.y = y + (size_t)t0 * c.H;
    cp.w = m->tcw;
    cp.T = Tg;
    cp.k = c.k;
    cp.H = c.H;
    const int G = m->num_sms;
    if (launch(moe::moe_tc_prep, dim3(std::min(G, P)), dim3(moe::kTcPrepThreads),
               moe::tc_prep_smem(P, c.E), s, pdl, pp) != cudaSuccess ||
        (m->tc_f16_gu
             ? launch(moe::moe_tc_gate_up<F, true>, dim3(G), dim3(moe::kTcGuThreads), m->tc_smem_gu,
                      s, pdl, gp)
             : launch(moe::moe_tc_gate_up<F, false>, dim3(G), dim3(moe::kTcGuThreads),
                      m->tc_smem_gu, s, pdl, gp)) != cudaSuccess ||
        launch(moe::moe_tc_down<F>, dim3(G), dim3(moe::kTcDnThreads), m->tc_smem_dn, s, pdl,
               dp) != cudaSuccess ||
        launch(moe::moe_tc_combine, dim3((c.H + 4 * moe::kTcCombineThreads - 1) /
                                             (4 * moe::kTcCombineThreads),
                                         Tg),
               dim3(moe::kTcCombineThreads), 0, s, pdl, cp) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status_t tc_layer(moe_decode* m, int T, const uint16_t* x, const int32_t* ids, const float* w,
                      uint16_t* h, uint16_t* y, cudaStream_t s) {
  return is_fp4(m) ? tc_layer_f<moe::TcFp4>(m, T, x, ids, w, h, y, s)
                   : tc_layer_f<moe::TcFp8>(m, T, x, ids, w, h, y, s);
}

// ---- per-call token chunking -----------------------------------------------

// Tokens per gate/up launch: groups of 32, or, when a group's x does not fit
// in shared memory (the kernel that reads x through L1 would run) but that of
// a group of at least four does, groups of the largest such size. Each group
// streams its unique experts once, so smaller groups read an expert shared
// between groups more than once; the staged kernel more than pays for that.
int gate_up_group(const moe_decode* m, int T) {
  int g = std::min(T, moe::kMaxTokensPerLaunch);
  int SG = 0;
  size_t smem = 0;
  if (g < 2 || gate_up_kind(m, g, SG, smem) != GuKind::kL1) return g;
  int g2 = g;
  while (g2 > 4 && moe::gate_up_xs_smem(g2, m->cfg.H, kmax_of(m)) > m->smem_per_block) --g2;
  if (moe::gate_up_xs_smem(g2, m->cfg.H, kmax_of(m)) > m->smem_per_block) return g;
  // equal groups: T = 16 with room for 15 runs as two groups of 8
  const int n = (T + g2 - 1) / g2;
  return (T + n - 1) / n;
}

moe_status_t gate_up_chunks(moe_decode* m, int T, const uint16_t* x, const int32_t* ids,
                            uint16_t* h, cudaStream_t s) {
  const moe_decode_config_t& c = m->cfg;
  const int G = gate_up_group(m, T);
  for (int t0 = 0; t0 < T; t0 += G) {
    moe::GateUpParams p;
    p.T = std::min(G, T - t0);
    p.x = x + (size_t)t0 * c.H;
    p.ids = ids + (size_t)t0 * c.k;
    p.h = h + (size_t)t0 * c.k * c.I;
    p.wgu = m->wgu;
    p.sgu = m->sgu;
    p.err = m->d_err;
    p.k = c.k;
    p.E = c.E;
    p.H = c.H;
    p.I = c.I;
    if (launch_gate_up(m, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status_t down_chunks(moe_decode* m, int T, const uint16_t* h, const int32_t* ids,
                         const float* w, uint16_t* y, bool early, cudaStream_t s) {
  const moe_decode_config_t& c = m->cfg;
  for (int t0 = 0; t0 < T; t0 += moe::kMaxTokensPerLaunch) {
    moe::DownParams p;
    p.T = std::min(moe::kMaxTokensPerLaunch, T - t0);
    p.h = h + (size_t)t0 * c.k * c.I;
    p.ids = ids + (size_t)t0 * c.k;
    p.w = w + (size_t)t0 * c.k;
    p.y = y + (size_t)t0 * c.H;
    p.wd = m->wd;
    p.sd = m->sd;
    p.err = m->d_err;
    p.k = c.k;
    p.E = c.E;
    p.H = c.H;
    p.I = c.I;
    p.early = early ? 1 : 0;
    if (launch_down(m, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// The layer's launches for T >= 1 tokens (arguments checked by the caller).
moe_status_t layer_enqueue(moe_decode* m, int T, const uint16_t* x, const int32_t* topk_ids,
                           const float* topk_w, uint16_t* h, uint16_t* y, cudaStream_t s) {
  if (use_tc(m, T)) return tc_layer(m, T, x, topk_ids, topk_w, h, y, s);
  if (T == 1 && m->fused_ok) return fused_layer(m, x, topk_ids, topk_w, h, y, s);
  moe_status_t st;
  if (T <= moe::kMaxTokensPerLaunch) {
    st = gate_up_chunks(m, T, x, topk_ids, h, s);
    if (st != MOE_OK) return st;
    return down_chunks(m, T, h, topk_ids, topk_w, y, use_pdl(m), s);
  }
  // several token groups: finish every gate/up launch before the downs so the
  // early weight fetch of a down never precedes a gate/up it does not follow
  st = gate_up_chunks(m, T, x, topk_ids, h, s);
  if (st != MOE_OK) return st;
  return down_chunks(m, T, h, topk_ids, topk_w, y, false, s);
}

moe_status_t check_T(const moe_decode* m, int32_t T) {
  if (!m) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > m->cfg.max_T) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Host-side checks of a layer call (T = 0 passes: a no-op).
moe_status_t check_layer(const moe_decode* m, int32_t T, const uint16_t* x, const int32_t* ids,
                         const float* w, const uint16_t* h, const uint16_t* y) {
  moe_status_t st = check_T(m, T);
  if (st != MOE_OK || T == 0) return st;
  if (!x || !ids || !w || !h || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 32) || !aligned(h, 32) || !aligned(ids, 4) || !aligned(w, 4) || !aligned(y, 2))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

// After a call has enqueued its work on s: record the handle's completion
// event there, unless s is being captured into a graph (the event would then
// stand for a graph node, not for work that runs).
void mark_done(moe_decode* m, cudaStream_t s) {
  if (!m->done_ev) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return;
  }
  if (cs != cudaStreamCaptureStatusNone) return;
  if (cudaEventRecord(m->done_ev, s) == cudaSuccess) m->done_recorded = true;
}

moe_status_t enqueued(moe_decode* m, cudaStream_t s, moe_status_t st) {
  if (st == MOE_OK) mark_done(m, s);
  return st;
}

// Read and clear the device error word on the handle's private stream (and,
// after a timeout, restart the one-launch kernel's counters from zero).
moe_status_t read_error(moe_decode* m, uint32_t* device_flags) {
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, m->d_err, sizeof(v), cudaMemcpyDeviceToHost, m->aux) != cudaSuccess ||
      cudaStreamSynchronize(m->aux) != cudaSuccess ||
      cudaMemsetAsync(m->d_err, 0, sizeof(v), m->aux) != cudaSuccess ||
      // a bounded wait that gave up may have left the launch and barrier
      // counters out of step: start both again from zero
      ((v & moe::kDeviceTimeout) && cudaMemsetAsync(m->d_bar, 0, 16, m->aux) != cudaSuccess) ||
      cudaStreamSynchronize(m->aux) != cudaSuccess)
    return MOE_ERR_CUDA;
  *device_flags = v;
  return v ? MOE_ERR_DEVICE_FAULT : MOE_OK;
}

void free_all(moe_decode* m) {
  if (!m) return;
  if (m->done_ev) cudaEventDestroy(m->done_ev);
  if (m->aux) cudaStreamDestroy(m->aux);
  cudaFree(m->d_err);
  cudaFree(m->d_x);
  cudaFree(m->d_ids);
  cudaFree(m->d_w);
  cudaFree(m->d_h);
  cudaFree(m->d_y);
  cudaFree(m->tc_mem);
  delete m;
}

}  // namespace

extern "C" {

moe_status_t moe_decode_create(const moe_decode_config_t* cfg, const uint8_t* w_gateup,
                               const uint8_t* s_gateup, const uint8_t* w_down,
                               const uint8_t* s_down, moe_decode_t* out) {
  if (out) *out = nullptr;
  if (!cfg || !out || !w_gateup || !s_gateup || !w_down || !s_down) return MOE_ERR_INVALID_ARG;
  const moe_decode_config_t c = *cfg;
  if (c.E < 1 || c.k < 1 || c.H < 1 || c.I < 1 || c.max_T < 0) return MOE_ERR_INVALID_ARG;
  if (c.k > c.E) return MOE_ERR_INVALID_ARG;
  if (c.E > kMaxE || c.k > kMaxK || c.H % 32 || c.I % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((c.flags & ~kKnownFlags) != 0) return MOE_ERR_INVALID_ARG;
  const size_t down_smem = (size_t)c.k * c.I * sizeof(float);
  if (down_smem > kMaxDownSmem) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w_gateup, 32) || !aligned(w_down, 32)) return MOE_ERR_MISALIGNED;

  moe_decode* m = new (std::nothrow) moe_decode();
  if (!m) return MOE_ERR_CUDA;
  m->cfg = c;
  m->wgu = w_gateup;
  m->sgu = s_gateup;
  m->wd = w_down;
  m->sd = s_down;
  m->down_smem = down_smem;
  bool ok = cudaGetDevice(&m->device) == cudaSuccess &&
            cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) ==
                cudaSuccess &&
            cudaMalloc(&m->d_err, 32) == cudaSuccess && cudaMemset(m->d_err, 0, 32) == cudaSuccess &&
            cudaEventCreateWithFlags(&m->done_ev, cudaEventDisableTiming) == cudaSuccess &&
            cudaStreamCreateWithFlags(&m->aux, cudaStreamNonBlocking) == cudaSuccess;
  if (ok) m->d_bar = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(m->d_err) + 8);
  int pageable = 0;
  ok = ok && cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, m->device) ==
                 cudaSuccess;
  m->host_direct = pageable != 0;
  ok = ok && query_fused(m);
  m->gu_tma_ok = ok && encode_gu_tma_maps(m);
  m->dn_tma_ok = ok && encode_dn_tma_maps(m);
  ok = ok && tc_setup(m);


  ok = ok && set_down_attributes() == cudaSuccess;
  int occ = 0;
  ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                 &occ, moe::moe_gate_up_3d_batched<1, 8, moe::Mxfp8>, moe::kThreads, 0) ==
                 cudaSuccess;
  m->gate_up_ctas_per_sm = std::max(1, occ);
  if (ok && c.max_T > 0) {
    const size_t T = (size_t)c.max_T;
    ok = cudaMalloc(&m->d_x, T * c.H * 2) == cudaSuccess &&
         cudaMalloc(&m->d_ids, T * c.k * 4) == cudaSuccess &&
         cudaMalloc(&m->d_w, T * c.k * 4) == cudaSuccess &&
         cudaMalloc(&m->d_h, T * c.k * c.I * 2) == cudaSuccess &&
         cudaMalloc(&m->d_y, T * c.H * 2) == cudaSuccess;
  }
  if (!ok) {
    free_all(m);
    return MOE_ERR_CUDA;
  }
  *out = m;
  return MOE_OK;
}

moe_status_t moe_decode_destroy(moe_decode_t m) {
  if (!m) return MOE_OK;
  free_all(m);
  return MOE_OK;
}

moe_status_t moe_route(moe_decode_t m, int32_t T, const float* logits, int32_t* topk_ids,
                       float* topk_w, void* stream) {
  moe_status_t st = check_T(m, T);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)) return MOE_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid((T + moe::kWarps - 1) / moe::kWarps), block(moe::kThreads);
  const int E = m->cfg.E, k = m->cfg.k;
  cudaError_t e;
  if (E <= 128)
    e = launch(moe::moe_route_topk<4>, grid, block, 0, s, use_pdl(m), logits, T, E, k, topk_ids, topk_w);
  else if (E <= 256)
    e = launch(moe::moe_route_topk<8>, grid, block, 0, s, use_pdl(m), logits, T, E, k, topk_ids, topk_w);
  else
    e = launch(moe::moe_route_topk<32>, grid, block, 0, s, use_pdl(m), logits, T, E, k, topk_ids, topk_w);
  return enqueued(m, s, e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA);
}

moe_status_t moe_dedup_schedule(moe_decode_t m, int32_t T, const int32_t* topk_ids, int32_t* uniq,
                                int32_t* offsets, int32_t* pairs, int32_t* n_uniq, void* stream) {
  moe_status_t st = check_T(m, T);
  if (st != MOE_OK) return st;
  if (T > moe::kMaxTokensPerLaunch) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !uniq || !offsets || !pairs || !n_uniq) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int E = m->cfg.E, k = m->cfg.k;
  cudaError_t e;
  if (k <= 8)
    e = launch(moe::moe_dedup_schedule_kernel<8>, dim3(1), dim3(32), 0, s, use_pdl(m), topk_ids, T,
               k, E, uniq, offsets, pairs, n_uniq, m->d_err);
  else
    e = launch(moe::moe_dedup_schedule_kernel<32>, dim3(1), dim3(32), 0, s, use_pdl(m), topk_ids,
               T, k, E, uniq, offsets, pairs, n_uniq, m->d_err);
  return enqueued(m, s, e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA);
}

moe_status_t moe_gate_up(moe_decode_t m, int32_t T, const uint16_t* x, const int32_t* topk_ids,
                         uint16_t* h, void* stream) {
  moe_status_t st = check_T(m, T);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x || !topk_ids || !h) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 32) || !aligned(h, 32) || !aligned(topk_ids, 4)) return MOE_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return enqueued(m, s, gate_up_chunks(m, T, x, topk_ids, h, s));
}

moe_status_t moe_down(moe_decode_t m, int32_t T, const uint16_t* h, const int32_t* topk_ids,
                      const float* topk_w, uint16_t* y, void* stream) {
  moe_status_t st = check_T(m, T);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!h || !topk_ids || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(h, 32) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(y, 2))
    return MOE_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return enqueued(m, s, down_chunks(m, T, h, topk_ids, topk_w, y, false, s));
}

moe_status_t moe_decode_layer(moe_decode_t m, int32_t T, const uint16_t* x,
                              const int32_t* topk_ids, const float* topk_w, uint16_t* h,
                              uint16_t* y, void* stream) {
  moe_status_t st = check_layer(m, T, x, topk_ids, topk_w, h, y);
  if (st != MOE_OK || T == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return enqueued(m, s, layer_enqueue(m, T, x, topk_ids, topk_w, h, y, s));
}

moe_status_t moe_decode_forward_host(moe_decode_t m, int32_t T, const uint16_t* x_host,
                                     const int32_t* ids_host, const float* w_host,
                                     uint16_t* y_host, void* stream) {
  moe_status_t st = check_T(m, T);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x_host || !ids_host || !w_host || !y_host) return MOE_ERR_INVALID_ARG;
  const moe_decode_config_t& c = m->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // host buffers the device can address are read and written by the kernels
  // in place, with no copy-engine round trips: any host memory on a device
  // that accesses pageable memory coherently (at the host's addresses), else
  // page-locked buffers through their device mapping
  const bool copy = (c.flags & MOE_FLAG_HOST_COPY) != 0;
  const void* xd = copy ? nullptr : m->host_direct ? x_host : mapped_host(x_host);
  const void* idd = copy ? nullptr : m->host_direct ? ids_host : mapped_host(ids_host);
  const void* wd = copy ? nullptr : m->host_direct ? w_host : mapped_host(w_host);
  void* yd = copy ? nullptr : m->host_direct ? y_host : const_cast<void*>(mapped_host(y_host));
  if (xd && idd && wd && yd) {
    // the stream is synchronised below, so no completion event is recorded
    const uint16_t* xp = static_cast<const uint16_t*>(xd);
    const int32_t* ip = static_cast<const int32_t*>(idd);
    const float* wp = static_cast<const float*>(wd);
    uint16_t* yp = static_cast<uint16_t*>(yd);
    st = check_layer(m, T, xp, ip, wp, m->d_h, yp);
    if (st == MOE_OK) st = layer_enqueue(m, T, xp, ip, wp, m->d_h, yp, s);
    if (st != MOE_OK) return st;
    return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (cudaMemcpyAsync(m->d_x, x_host, (size_t)T * c.H * 2, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(m->d_ids, ids_host, (size_t)T * c.k * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(m->d_w, w_host, (size_t)T * c.k * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = layer_enqueue(m, T, m->d_x, m->d_ids, m->d_w, m->d_h, m->d_y, s);
  if (st != MOE_OK) return st;
  if (cudaMemcpyAsync(y_host, m->d_y, (size_t)T * c.H * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_decode_get_error(moe_decode_t m, uint32_t* device_flags) {
  if (!m || !device_flags) return MOE_ERR_INVALID_ARG;
  // only the handle's own latest call is waited for: work of other streams
  // and other libraries keeps running
  if (m->done_recorded && cudaEventSynchronize(m->done_ev) != cudaSuccess) return MOE_ERR_CUDA;
  return read_error(m, device_flags);
}

moe_status_t moe_decode_get_error_stream(moe_decode_t m, void* stream, uint32_t* device_flags) {
  if (!m || !device_flags) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  return read_error(m, device_flags);
}

const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_FAULT: return "device flagged an error";
  }
  return "unknown status";
}

int32_t moe_decode_version(void) { return kVersion; }

int32_t moe_decode_fused_layer(moe_decode_t m) { return m ? (m->fused_ok ? 1 : 0) : -1; }

moe_status_t moe_decode_set_path(moe_decode_t m, int32_t path) {
  if (!m || path < MOE_PATH_AUTO || path > MOE_PATH_TENSOR) return MOE_ERR_INVALID_ARG;
  if (path == MOE_PATH_TENSOR && !m->tc_ok) return MOE_ERR_UNSUPPORTED_SHAPE;
  m->path = path;
  return MOE_OK;
}

int32_t moe_decode_path(moe_decode_t m, int32_t T) {
  if (!m || T < 1) return -1;
  return use_tc(m, T) ? MOE_PATH_TENSOR : MOE_PATH_WARP;
}

int32_t moe_decode_tensor_path(moe_decode_t m) { return m ? (m->tc_ok ? 1 : 0) : -1; }

moe_status_t moe_decode_plan(const moe_decode_config_t* cfg, int32_t num_sms,
                             int32_t smem_per_block, int32_t T, moe_decode_plan_t* out) {
  if (!cfg || !out || num_sms < 1 || smem_per_block < 1 || T < 1) return MOE_ERR_INVALID_ARG;
  const moe_decode_config_t c = *cfg;
  if (c.E < 1 || c.k < 1 || c.H < 1 || c.I < 1 || c.k > c.E) return MOE_ERR_INVALID_ARG;
  if (c.E > kMaxE || c.k > kMaxK || c.H % 32 || c.I % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((c.flags & ~kKnownFlags) != 0) return MOE_ERR_INVALID_ARG;
  // a handle on the stack with 256-byte aligned stand-in weight pointers
  // (never dereferenced) and the given device limits
  moe_decode m = {};
  m.cfg = c;
  m.wgu = m.sgu = m.wd = m.sd = reinterpret_cast<const uint8_t*>(uintptr_t{256});
  m.num_sms = num_sms;
  m.smem_per_block = (size_t)smem_per_block;
  m.fused_ok = true;
  m.gu_tma_ok = gu_tma_shape_ok(&m);
  m.dn_tma_ok = dn_tma_shape_ok(&m);
  *out = moe_decode_plan_t{};
  moe::FusedParams fp = {};
  size_t smem = 0;
  if (plan_fused(&m, fp, smem)) {
    out->fused = 1;
    out->fused_kc = fp.KC;
    out->fused_slots = fp.SG;
    out->fused_slot_bytes = fp.slot_g;
    out->fused_down_rows = fp.RC;
    out->fused_down_per_slot = fp.SR;
    out->fused_smem = (int32_t)smem;
  }
  const int G = gate_up_group(&m, T);
  int SG = 0;
  smem = 0;
  out->gate_up_group = G;
  const GuKind gk = gate_up_kind(&m, G, SG, smem);
  out->gate_up_kernel = gk == GuKind::kL1 ? 0 : gk == GuKind::kXs ? 1 : 2;
  out->gate_up_slots = gk == GuKind::kTma ? SG : 0;
  out->gate_up_smem = gk == GuKind::kL1 ? 0 : (int32_t)smem;
  SG = 0;
  smem = 0;
  const DnKind dk = down_kind(&m, std::min<int>(T, moe::kMaxTokensPerLaunch), SG, smem);
  out->down_kernel = dk == DnKind::kWarp ? 0 : dk == DnKind::kTma ? 1 : 2;
  out->down_slots = dk == DnKind::kWarp ? 0 : SG;
  out->down_smem = (int32_t)smem;
  return MOE_OK;
}

const char* moe_decode_kernel_name(moe_decode_t m, int32_t T, int32_t which) {
  if (!m || T <= 0 || (which != 0 && which != 1)) return "";
  if (use_tc(m, T)) return which == 0 ? "moe_tc_gate_up" : "moe_tc_down";
  const int Tl = std::min<int>(T, moe::kMaxTokensPerLaunch);
  int SG = 0;
  size_t smem = 0;
  if (which == 0) {
    switch (gate_up_kind(m, gate_up_group(m, T), SG, smem)) {
      case GuKind::kTma: return "moe_gate_up_tma";
      case GuKind::kXs: return "moe_gate_up_3d_batched_xs";
      case GuKind::kL1: return "moe_gate_up_3d_batched";
    }
    return "";
  }
  switch (down_kind(m, Tl, SG, smem)) {
    case DnKind::kMma: return "moe_down_mma";
    case DnKind::kTma: return "moe_down_tma";
    case DnKind::kWarp: return "moe_down_3d_batched";
  }
  return "";
}

moe_status_t moe_decode_arm_barrier_timeout(moe_decode_t m) {
  if (!m) return MOE_ERR_INVALID_ARG;
  if (!m->fused_ok) return MOE_ERR_UNSUPPORTED_SHAPE;
  // 0x0101...01: a launch index no barrier count of this handle can reach
  if (cudaMemset(m->d_bar, 0x01, 8) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

#ifdef MOE_TIMELINE
moe_status_t moe_decode_layer_timeline(moe_decode_t m, const uint16_t* x, const int32_t* topk_ids,
                                       const float* topk_w, uint16_t* h, uint16_t* y,
                                       uint64_t* stamps, void* stream) {
  moe_status_t st = check_layer(m, 1, x, topk_ids, topk_w, h, y);
  if (st != MOE_OK) return st;
  if (!stamps || !aligned(stamps, 8)) return MOE_ERR_INVALID_ARG;
  if (!m->fused_ok) return MOE_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return enqueued(m, s, fused_layer(m, x, topk_ids, topk_w, h, y, s,
                                    reinterpret_cast<unsigned long long*>(stamps)));
}

int32_t moe_decode_timeline_ctas(moe_decode_t m) { return m ? m->num_sms : -1; }
#endif

}  // extern "C"

// ---------------------------------------------------------------------------
// The layer without device allocation (moe_decode_layer_noalloc).
//
// For callers that cannot call cudaMalloc: h and the error word live in one
// file-scope array of static device memory. In host code the array's name is
// only a stand-in for the device object, so its device address is looked up
// with cudaGetSymbolAddress once per device (with that device current) and
// that address is what the kernels receive.
// ---------------------------------------------------------------------------

namespace {

constexpr size_t kNoAllocHBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxDevices = 64;

// [0, kNoAllocHBytes): h of the current call; then the 4-byte error word and,
// 8 and 16 bytes on, the fused kernel's launch and grid-barrier counters.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocHBytes + 256];

struct NoAllocDevice {
  bool ready;
  uint8_t* scratch;   // device address of g_noalloc_scratch on this device
  int num_sms;
  int gate_up_ctas_per_sm;
  size_t smem_per_block;
  bool coop;          // the device supports cooperative launches
  // the plan and tensor maps of the latest configuration and weight pointers
  // seen on this device, reused while they stay the same
  bool have_plan;
  moe_decode plan;
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// One-time set-up for the current device: the array's device address, the
// SM count, the gate/up occupancy and the down kernel's shared-memory limit.
moe_status_t noalloc_device(int dev, NoAllocDevice* out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return MOE_ERR_CUDA;
    int occ = 0, coop = 0;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
        set_down_attributes() != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &occ, moe::moe_gate_up_3d_batched<1, 8, moe::Mxfp8>, moe::kThreads, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.scratch = static_cast<uint8_t*>(ptr);
    d.gate_up_ctas_per_sm = std::max(1, occ);
    moe_decode probe = {};
    probe.device = dev;
    probe.num_sms = d.num_sms;
    probe.cfg.k = 1;
    if (!query_fused(&probe)) return MOE_ERR_CUDA;
    d.smem_per_block = probe.smem_per_block;
    d.coop = coop != 0;
    d.have_plan = false;
    d.ready = true;
  }
  *out = d;
  return MOE_OK;
}

bool same_config(const moe_decode_config_t& a, const moe_decode_config_t& b) {
  return a.E == b.E && a.k == b.k && a.H == b.H && a.I == b.I && a.flags == b.flags;
}

// The stack handle of a call: launch plan, kernel choices and tensor maps for
// this configuration and these weights, taken from the device's cache when
// the previous call used the same ones, else planned and cached.
void noalloc_plan(int dev, const NoAllocDevice& d, const moe_decode_config_t& c,
                  const uint8_t* wgu, const uint8_t* sgu, const uint8_t* wd, const uint8_t* sd,
                  moe_decode* m) {
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    const NoAllocDevice& cached = g_noalloc_dev[dev];
    if (cached.have_plan && same_config(cached.plan.cfg, c) && cached.plan.wgu == wgu &&
        cached.plan.sgu == sgu && cached.plan.wd == wd && cached.plan.sd == sd) {
      *m = cached.plan;
      return;
    }
  }
  *m = moe_decode{};
  m->cfg = c;
  m->wgu = wgu;
  m->sgu = sgu;
  m->wd = wd;
  m->sd = sd;
  m->device = dev;
  m->num_sms = d.num_sms;
  m->gate_up_ctas_per_sm = d.gate_up_ctas_per_sm;
  m->down_smem = (size_t)c.k * c.I * sizeof(float);
  m->smem_per_block = d.smem_per_block;
  {
    // the one-launch kernel: a cooperative launch whose plan depends on the shape
    moe::FusedParams fp = {};
    size_t smem = 0;
    m->fused_ok = d.coop;
    int occ = 0;
    const void* fk = is_fp4(m) ? (const void*)moe::moe_layer_fused_t1<8, moe::Mxfp4>
                               : (const void*)moe::moe_layer_fused_t1<8, moe::Mxfp8>;
    m->fused_ok = m->fused_ok && plan_fused(m, fp, smem) &&
                  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fk, moe::kFusedThreads,
                                                                smem) == cudaSuccess &&
                  occ >= 1 && encode_fused_maps(m, fp.KC, fp.RC);
  }
  m->gu_tma_ok = encode_gu_tma_maps(m);
  m->dn_tma_ok = encode_dn_tma_maps(m);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  g_noalloc_dev[dev].plan = *m;
  g_noalloc_dev[dev].have_plan = true;
}

}  // namespace

extern "C" moe_status_t moe_decode_layer_noalloc(const moe_decode_config_t* cfg,
                                                 const uint8_t* w_gateup, const uint8_t* s_gateup,
                                                 const uint8_t* w_down, const uint8_t* s_down,
                                                 int32_t T, const uint16_t* x,
                                                 const int32_t* topk_ids, const float* topk_w,
                                                 uint16_t* y, void* stream) {
  if (!cfg || !w_gateup || !s_gateup || !w_down || !s_down) return MOE_ERR_INVALID_ARG;
  const moe_decode_config_t c = *cfg;
  if (c.E < 1 || c.k < 1 || c.H < 1 || c.I < 1 || T < 0) return MOE_ERR_INVALID_ARG;
  if (c.k > c.E) return MOE_ERR_INVALID_ARG;
  if (c.E > kMaxE || c.k > kMaxK || c.H % 32 || c.I % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((c.flags & ~kKnownFlags) != 0) return MOE_ERR_INVALID_ARG;
  if ((size_t)c.k * c.I * sizeof(float) > kMaxDownSmem) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((size_t)T * c.k * c.I * 2 > kNoAllocHBytes) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w_gateup, 32) || !aligned(w_down, 32)) return MOE_ERR_MISALIGNED;
  if (T == 0) return MOE_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  NoAllocDevice d;
  const moe_status_t st = noalloc_device(dev, &d);
  if (st != MOE_OK) return st;
  // a handle on the stack: every device pointer in it is either the caller's
  // or inside the static array, and it has no staging buffers, event or stream
  moe_decode m;
  noalloc_plan(dev, d, c, w_gateup, s_gateup, w_down, s_down, &m);
  m.cfg.max_T = T;
  m.d_err = reinterpret_cast<uint32_t*>(d.scratch + kNoAllocHBytes);
  m.d_bar = reinterpret_cast<unsigned long long*>(d.scratch + kNoAllocHBytes + 8);
  return moe_decode_layer(&m, T, x, topk_ids, topk_w, reinterpret_cast<uint16_t*>(d.scratch), y,
                          stream);
}
