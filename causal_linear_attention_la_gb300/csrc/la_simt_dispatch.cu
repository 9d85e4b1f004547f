// Segment scan kernel and the head-size dispatch of the CUDA-core kernels.
#include "la_internal.cuh"

namespace la {

cudaError_t simt_segment_state_dk16(const FwdArgs&);
cudaError_t simt_segment_state_dk32(const FwdArgs&);
cudaError_t simt_segment_state_dk64(const FwdArgs&);
cudaError_t simt_segment_state_dk128(const FwdArgs&);
cudaError_t simt_forward_output_dk16(const FwdArgs&);
cudaError_t simt_forward_output_dk32(const FwdArgs&);
cudaError_t simt_forward_output_dk64(const FwdArgs&);
cudaError_t simt_forward_output_dk128(const FwdArgs&);
cudaError_t simt_backward_dk16(const BwdArgs&);
cudaError_t simt_backward_dk32(const BwdArgs&);
cudaError_t simt_backward_dk64(const BwdArgs&);
cudaError_t simt_backward_dk128(const BwdArgs&);

namespace {

// Segment scan over P records of `words` floats per (b,h): exclusive prefix
// (forward), exclusive suffix (reverse) or the total written into every slot.
// The inclusive total goes to S_final / z_final when given. Each thread owns
// 4 consecutive words (records are 16-byte multiples) and issues its loads in
// batches of 8 records before using them, so the dependent-latency chain is
// P / 8 loads long rather than P.
// With decay gating (alpha: per-head factors, else null; exclusive modes) the
// running sum decays by alpha^L_p across segment p of L_p tokens: forward
// records hold a segment's sums decayed to its last token, reverse records
// decayed to its first, so that slot p receives the state at segment p's
// start (forward) or the adjoint at the token after its end (reverse).
__global__ void scan_kernel(float* __restrict__ ws, int P, long long words,
                            int mode, float* __restrict__ S_final,
                            float* __restrict__ z_final, int dkdv, int dk,
                            const float* __restrict__ alpha, int H, int seg_len, int N) {
  const long long e = 4 * ((long long)blockIdx.y * blockDim.x + threadIdx.x);
  if (e >= words) return;
  const long long bh = blockIdx.x;
  float4* base = reinterpret_cast<float4*>(ws + bh * P * words + e);
  const long long stride = words / 4;   // in float4
  constexpr int BATCH = 8;
  float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [](float4& a, const float4& b) { a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w; };
  if (mode == SCAN_TOTAL) {
    for (int p0 = 0; p0 < P; p0 += BATCH) {
      float4 x[BATCH];
#pragma unroll
      for (int i = 0; i < BATCH; ++i) x[i] = p0 + i < P ? base[(p0 + i) * stride] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < BATCH; ++i) add(run, x[i]);
    }
    for (int p = 0; p < P; ++p) base[p * stride] = run;
  } else {
    const bool rev = mode == SCAN_EXCLUSIVE_REV;
    const float log2a = alpha != nullptr ? log2f(alpha[bh % H]) : 0.f;
    for (int p0 = 0; p0 < P; p0 += BATCH) {
      float4 x[BATCH];
#pragma unroll
      for (int i = 0; i < BATCH; ++i) {
        const int p = rev ? P - 1 - (p0 + i) : p0 + i;
        x[i] = p0 + i < P ? base[p * stride] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < BATCH; ++i) {
        const int p = rev ? P - 1 - (p0 + i) : p0 + i;
        if (p0 + i < P) {
          base[p * stride] = run;
          if (alpha != nullptr) {
            // segment p's tokens decay what the running sum carries past it
            const float f = exp2f((float)min(seg_len, N - p * seg_len) * log2a);
            run.x *= f; run.y *= f; run.z *= f; run.w *= f;
          }
        }
        add(run, x[i]);
      }
    }
  }
  if (S_final != nullptr) {
    const float v[4] = {run.x, run.y, run.z, run.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long ej = e + j;
      if (ej < dkdv) S_final[bh * dkdv + ej] = v[j];
      else z_final[bh * dk + (ej - dkdv)] = v[j];
    }
  }
}

}  // namespace

cudaError_t simt_segment_state(const FwdArgs& a) {
  switch (a.dk) {
    case 16: return simt_segment_state_dk16(a);
    case 32: return simt_segment_state_dk32(a);
    case 64: return simt_segment_state_dk64(a);
    case 128: return simt_segment_state_dk128(a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t simt_forward_output(const FwdArgs& a) {
  switch (a.dk) {
    case 16: return simt_forward_output_dk16(a);
    case 32: return simt_forward_output_dk32(a);
    case 64: return simt_forward_output_dk64(a);
    case 128: return simt_forward_output_dk128(a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t simt_backward(const BwdArgs& a) {
  switch (a.dk) {
    case 16: return simt_backward_dk16(a);
    case 32: return simt_backward_dk32(a);
    case 64: return simt_backward_dk64(a);
    case 128: return simt_backward_dk128(a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t segment_scan(float* ws, int BH, int P, long long words, int mode,
                         float* S_final, float* z_final, int dk, int dv,
                         cudaStream_t stream, const float* alpha, int H, int seg_len, int N) {
  // records of dk*dv + dk floats: always a multiple of 4 (dk >= 16)
  dim3 grid(BH, (unsigned)((words / 4 + 255) / 256));
  scan_kernel<<<grid, 256, 0, stream>>>(ws, P, words, mode, S_final, z_final,
                                        dk * dv, dk, alpha, H, seg_len, N);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace la
