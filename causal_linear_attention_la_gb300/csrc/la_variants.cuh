// Declarations of the state-update variants (decay gating, delta rule) and the
// state copy; host launchers defined in la_variants.cu.
#pragma once

#include <cuda_runtime.h>

#include "la.h"

namespace la {

struct VariantArgs {
  float* S; float* z;                 // state (z unused by the delta rule)
  const void* q; const void* k; const void* v; void* out;
  const float* alpha;                 // decay: [H] per-head factors (device)
  int H, BH, ntok, dk, dv; float eps; la_dtype dtype;
  cudaStream_t stream;
};

cudaError_t decode_steps_decay(const VariantArgs& a);
cudaError_t decode_steps_delta(const VariantArgs& a);
// Delta rule over whole sequences in 32-token chunks (la_delta_fwd.cu):
// ntok = N tokens per (batch, head), dk = dv in {16, 32, 64, 128}.
cudaError_t forward_delta_chunked(const VariantArgs& a);
// Decay-gated causal forward on the tensor cores (bf16, dk = dv = 64): the
// state pass and the chunk loop with per-head factors alpha [H]; FwdArgs as
// for la_forward (its segment plan and workspace).
struct FwdArgs;
cudaError_t tc_forward_decay(const FwdArgs& a, const float* alpha, int H);
// The tensor-core multi-token decode with decay gating (la_decode_tc.cu;
// where tc_decode_supported holds): per-head factors alpha [H] (device).
struct DecodeArgs;
cudaError_t tc_decode_steps_decay(const DecodeArgs& a, const float* alpha, int H);
// ... and the delta rule (S only; no z)
cudaError_t tc_decode_steps_delta(const DecodeArgs& a);
// dst <- src for n floats (16-byte aligned pointers)
cudaError_t copy_floats(float* dst, const float* src, long long n, cudaStream_t stream);

}  // namespace la
