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
// The inclusive total goes to S_final / z_final when given.
__global__ void scan_kernel(float* __restrict__ ws, int P, long long words,
                            int mode, float* __restrict__ S_final,
                            float* __restrict__ z_final, int dkdv, int dk) {
  const long long e = (long long)blockIdx.y * blockDim.x + threadIdx.x;
  if (e >= words) return;
  const long long bh = blockIdx.x;
  float* base = ws + bh * P * words + e;
  float run = 0.f;
  if (mode == SCAN_TOTAL) {
    for (int p = 0; p < P; ++p) run += base[p * words];
    for (int p = 0; p < P; ++p) base[p * words] = run;
  } else if (mode == SCAN_EXCLUSIVE_FWD) {
    for (int p = 0; p < P; ++p) {
      const float x = base[p * words];
      base[p * words] = run;
      run += x;
    }
  } else {
    for (int p = P - 1; p >= 0; --p) {
      const float x = base[p * words];
      base[p * words] = run;
      run += x;
    }
  }
  if (S_final != nullptr) {
    if (e < dkdv) S_final[bh * dkdv + e] = run;
    else z_final[bh * dk + (e - dkdv)] = run;
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
                         cudaStream_t stream) {
  dim3 grid(BH, (unsigned)((words + 255) / 256));
  scan_kernel<<<grid, 256, 0, stream>>>(ws, P, words, mode, S_final, z_final,
                                        dk * dv, dk);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace la
