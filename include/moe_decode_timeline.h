/*
 * moe_decode_timeline.h -- the per-CTA timeline of the one-launch single-token
 * layer, in libmoe_decode_timeline.so only: the same sources as
 * libmoe_decode.so compiled with -DMOE_TIMELINE (the package's build script
 * makes it with `python -m sparse_expert_gemv_gb300.build --timeline`). It
 * exports every entry point of moe_decode.h plus the two below. The pages
 * have no counterpart: it is a measurement aid that shows where the time of
 * the one-launch kernel goes, phase by phase and CTA by CTA.
 */
#ifndef MOE_DECODE_TIMELINE_H
#define MOE_DECODE_TIMELINE_H

#include <stdint.h>

#include "moe_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Stamps per CTA and their meaning; each is the GPU's global nanosecond timer
 * (%globaltimer) read when that CTA reaches the point. */
#define MOE_TL_STAMPS 16
enum {
  MOE_TL_ENTRY = 0,          /* kernel entry */
  MOE_TL_INPUTS = 1,         /* programmatic-dependence wait passed: inputs readable */
  MOE_TL_ROUTED = 2,         /* routing ids read and the expert schedule built (producer warp) */
  MOE_TL_FIRST_ISSUE = 3,    /* first weight tile issued (producer warp) */
  MOE_TL_FIRST_LANDED = 4,   /* first weight tile landed (consumer warps) */
  MOE_TL_GATE_UP_DONE = 5,   /* the CTA's gate/up tiles reduced and its h stored */
  MOE_TL_ARRIVING = 6,       /* about to post the CTA's grid-barrier arrival */
  MOE_TL_DOWN_LANDED = 7,    /* the first down row chunk's rows landed */
  MOE_TL_BARRIER = 8,        /* grid barrier passed: every CTA's h is written */
  MOE_TL_H_STAGED = 9,       /* h read back and staged in shared memory */
  MOE_TL_DOWN_DONE = 10,     /* the CTA's rows of y reduced and stored */
  MOE_TL_ISSUE_DONE = 11     /* the CTA's last weight tile issued */
};

/*
 * moe_decode_layer with T = 1 through the one-launch kernel, which also writes
 * MOE_TL_STAMPS uint64 stamps per CTA to `stamps` (device, 8-byte aligned,
 * moe_decode_timeline_ctas(handle) * MOE_TL_STAMPS entries; stamps a CTA does
 * not reach are left unchanged). Returns MOE_ERR_UNSUPPORTED_SHAPE when the
 * handle's single-token layer does not run as one launch
 * (moe_decode_fused_layer), otherwise as moe_decode_layer.
 */
moe_status_t moe_decode_layer_timeline(moe_decode_t handle, const uint16_t* x,
                                       const int32_t* topk_ids, const float* topk_w,
                                       uint16_t* h, uint16_t* y, uint64_t* stamps,
                                       void* stream);

/* CTAs of the one-launch kernel on this handle's device (rows of `stamps`), -1 for NULL. */
int32_t moe_decode_timeline_ctas(moe_decode_t handle);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_TIMELINE_H */
