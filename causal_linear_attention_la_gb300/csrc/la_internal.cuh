// Internal declarations shared by the host entry points and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "la.h"

namespace la {

// ---------------------------------------------------------------------------
// Feature map phi(x) = elu(x) + 1: x + 1 for x >= 0, exp(x) for x < 0
// ("Transformers are RNNs" review, feature-map table). For x < 0,
// elu(x) + 1 = exp(x) - 1 + 1 = exp(x), evaluated directly so that it stays
// positive and accurate for very negative x.
// phi'(x) = 1 for x >= 0 and exp(x) for x < 0, i.e. min(phi(x), 1).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float phi(float x) { return x >= 0.f ? x + 1.f : expf(x); }
__device__ __forceinline__ float phi_prime_from_phi(float p) { return fminf(p, 1.f); }

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

constexpr int kSegGranuleDecl = 128;  // = kSegGranule (declared below)

// ---------------------------------------------------------------------------
// Sequence segmentation: each (batch, head) sequence is cut into P segments
// of seg_len tokens (the last may be shorter); one CTA per (segment, b*h).
// ---------------------------------------------------------------------------
struct SegPlan {
  int P;        // segments per sequence (>= 1)
  int seg_len;  // tokens per segment, multiple of kSegGranule (except when N is smaller)
  int F = 1;    // tensor-core state pass: CTAs (and sum records) per segment
  // Balanced pieces (NP > 0; the causal tensor-core forward at d = 128 without
  // a final state): the heads' chunks laid end to end, head after head, and
  // cut into NP pieces of piece_len chunks (the last one shorter), one CTA
  // each; a piece may end one head and start the next. Record i is the sum
  // over the part of piece i in its last head, when that head goes on after
  // the piece. P and seg_len still describe the segment plan.
  int NP = 0;
  int piece_len = 0;
};

// Tokens summed by one state-pass CTA: ceil(chunks per segment / F) chunks.
inline int state_sub_len(const SegPlan& p) {
  const int L = (p.seg_len + kSegGranuleDecl - 1) / kSegGranuleDecl;
  return ((L + p.F - 1) / p.F) * kSegGranuleDecl;
}

constexpr int kSegGranule = kSegGranuleDecl;   // tokens; one tensor-core chunk
constexpr int kSlots = 152;        // CTAs resident at once: one per SM of a GB300

// Segments per sequence for B*H sequences of N tokens when `slots` CTAs can
// be resident at once.
SegPlan plan_segments(long long BH, int N, int slots = kSlots);

// Floats per per-segment state record of the CUDA-core kernels: dk*dv matrix
// then dk vector.
inline long long state_words(int dk, int dv) { return (long long)dk * dv + dk; }

// Floats reserved per record in the workspace: the tensor-core kernels' record
// (dk*dv matrix, dk vector, dv vector) is the larger of the two layouts.
inline long long record_slot_words(int dk, int dv) { return (long long)dk * dv + dk + dv; }

// ---------------------------------------------------------------------------
// Launchers (return cudaError_t of the launch; enqueue only)
// ---------------------------------------------------------------------------
struct FwdArgs {
  const void* q; const void* k; const void* v; void* out;
  int BH, N, dk, dv, causal; float eps; la_dtype dtype;
  float* S_final; float* z_final;
  float* ws_state;  // [BH][P][dk*dv + dk]
  SegPlan plan;
  cudaStream_t stream;
  // decay gating on the CUDA-core state pass: per-head factors [H] or null
  const float* alpha = nullptr;
  int H = 1;
};

struct BwdArgs {
  const void* q; const void* k; const void* v; const void* dout;
  void* dq; void* dk_; void* dv_;
  int BH, N, dk, dv, causal; float eps; la_dtype dtype;
  float* ws_state;  // [BH][P][dk*dv + dk]  forward state sums -> prefixes
  float* ws_rev;    // [BH][P][dk*dv + dk]  reverse sums (R, r) -> suffixes
  float* ws_tok;    // [BH][N][2]           D_t and b_t per token
  SegPlan plan;
  cudaStream_t stream;
  // ws_state already holds the forward's state-pass records (plan.F parts per
  // segment, as la_forward's tensor-core path leaves them): no state pass
  bool state_ready = false;
  // decay gating (CUDA-core path, causal): per-head factors [H] or null
  const float* alpha = nullptr;
  int H = 1;
};

struct DecodeArgs {
  float* S; float* z; const void* q; const void* k; const void* v; void* out;
  int BH, dk, dv; float eps; la_dtype dtype;
  cudaStream_t stream;
  int ntok = 1;     // tokens per (b,h) in this call (q, k, v, out hold ntok rows each)
};

// CUDA-core kernels (any supported head size, f32 or bf16)
cudaError_t simt_segment_state(const FwdArgs& a);                 // per-segment (dS, dz)
cudaError_t segment_scan(float* ws, int BH, int P, long long words,
                         int mode, float* S_final, float* z_final,
                         int dk, int dv, cudaStream_t stream,
                         const float* alpha = nullptr, int H = 1,
                         int seg_len = 0, int N = 0);               // prefix / suffix / total
cudaError_t simt_forward_output(const FwdArgs& a);
cudaError_t simt_backward(const BwdArgs& a);
cudaError_t decode_step(const DecodeArgs& a);
// tensor-core multi-token decode (bf16, dk = dv = 128, two tokens or more)
bool tc_decode_supported(int dk, int dv, la_dtype dtype, int ntok);
cudaError_t tc_decode_steps(const DecodeArgs& a);

// Tensor-core kernels (bf16, dk = dv in {64, 128}; causal and non-causal)
bool tc_forward_supported(int dk, int dv, la_dtype dtype, int causal);
cudaError_t tc_segment_state(const FwdArgs& a);
cudaError_t tc_forward_output(const FwdArgs& a);
// Tensor-core backward (bf16, dk = dv = 64, causal): state pass, scan, two sweeps
bool tc_backward_supported(int dk, int dv, la_dtype dtype, int causal);
cudaError_t tc_backward(const BwdArgs& a);

// Device status word of the current device (set to LA_ERR_TIMEOUT by a
// kernel whose bounded wait gave up); NULL if it cannot be resolved.
int* device_status_ptr();
// One-shot test switch (la_test_timeout_next_forward): true once after the
// switch is set, then false until it is set again.
bool take_timeout_test();

// Record a one-line reason for `s` as this thread's la_last_error; returns s.
la_status set_error(la_status s, const char* msg);

// scan modes
enum { SCAN_EXCLUSIVE_FWD = 0, SCAN_EXCLUSIVE_REV = 1, SCAN_TOTAL = 2 };

// Measurement hooks (la_profile_enable / la_profile_read / la_launch_count):
// prof_begin/prof_end record CUDA events around a span of launches on
// `stream` when profiling is on; note_launch counts kernel launches.
void prof_begin(int label, cudaStream_t stream);
void prof_end(int label, cudaStream_t stream);
void note_launch(int n = 1);

}  // namespace la
