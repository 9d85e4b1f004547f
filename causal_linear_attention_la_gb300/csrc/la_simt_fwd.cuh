// CUDA-core forward kernels: per-segment state sums and the chunked output
// kernel, instantiated for one key head size LA_DK per translation unit. These serve fp32 inputs and every head size; the
// tensor-core kernels take over for bf16 at the sizes they cover.
//
// Formulation (a re-association of the sums of "상태공간모델·선형 어텐션 —
// 어텐션의 O(N²) 대안", section 2, justified by the distributivity argument of
// "Linear Attention: KV를 고정 크기 상태에 누적하기", fig. 5): for a tile of TT
// tokens starting after state S_prev, z_prev,
//   num_t = phi(q_t)^T S_prev + sum_{j<=t in tile} (phi(q_t).phi(k_j)) v_j
//   den_t = phi(q_t).z_prev  + sum_{j<=t in tile}  phi(q_t).phi(k_j)  + eps
//   S    += sum_{j in tile} phi(k_j) v_j^T,  z += sum_j phi(k_j)
// Segments of one sequence start from the exclusive prefix of the per-segment
// sums, produced by segment_scan.
#include "la_internal.cuh"

#ifndef LA_DK
#error "define LA_DK before including this file"
#endif

namespace la {

namespace {

constexpr int NT = 256;  // threads per CTA
constexpr int TT = 32;   // tokens per tile

template <typename T>
__device__ __forceinline__ float ld(const T* p) { return to_f32<T>(*p); }

// Per-segment sums dS = sum phi(k) v^T, dz = sum phi(k) -> ws[bh][p]. With
// decay gating (alpha: per-head factors, else null) each token's term is
// weighted alpha^(last - token), the segment's sums decayed to its last token.
template <int DK, int DV, typename T>
__global__ void __launch_bounds__(NT)
simt_state_kernel(const T* __restrict__ k, const T* __restrict__ v, int N,
                  int P, int seg_len, float* __restrict__ ws,
                  const float* __restrict__ alpha, int H) {
  constexpr int RG = NT / DV;  // row groups
  constexpr int E = DK / RG;   // S rows per thread
  static_assert(E >= 1, "head size too small for this thread layout");
  __shared__ float fk[TT][DK + 1];
  __shared__ float vv[TT][DV];
  const long long bh = blockIdx.x;
  const int p = blockIdx.y;
  const int t0 = p * seg_len;
  const int t1 = min(N, t0 + seg_len);
  const T* kb = k + bh * N * DK;
  const T* vb = v + bh * N * DV;
  const int tid = threadIdx.x;
  const int m = tid % DV;
  const int c0 = tid / DV;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float zacc = 0.f;
  const float log2a = alpha != nullptr ? log2f(alpha[bh % H]) : 0.f;
  for (int s = t0; s < t1; s += TT) {
    const int n = min(TT, t1 - s);
    for (int idx = tid; idx < TT * DK; idx += NT) {
      const int t = idx / DK, c = idx % DK;
      fk[t][c] = t < n ? phi(ld(kb + (long long)(s + t) * DK + c)) * exp2f((float)(t1 - 1 - s - t) * log2a) : 0.f;
    }
    for (int idx = tid; idx < TT * DV; idx += NT) {
      const int t = idx / DV, c = idx % DV;
      vv[t][c] = t < n ? ld(vb + (long long)(s + t) * DV + c) : 0.f;
    }
    __syncthreads();
    for (int t = 0; t < n; ++t) {
      const float vm = vv[t][m];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(fk[t][c0 + e * RG], vm, acc[e]);
    }
    if (tid < DK)
      for (int t = 0; t < n; ++t) zacc += fk[t][tid];
    __syncthreads();
  }
  float* o = ws + (bh * P + p) * (long long)(DK * DV + DK);
#pragma unroll
  for (int e = 0; e < E; ++e) o[(c0 + e * RG) * DV + m] = acc[e];
  if (tid < DK) o[DK * DV + tid] = zacc;
}

template <int DK, int DV>
constexpr size_t output_smem_bytes() {
  return sizeof(float) * (size_t)(DK * DV + DK + 2 * TT * (DK + 1) + TT * DV +
                                  TT * (TT + 1) + TT);
}

// Chunked output for one segment, starting from the prefix state in ws.
template <int DK, int DV, typename T>
__global__ void __launch_bounds__(NT)
simt_output_kernel(const T* __restrict__ q, const T* __restrict__ k,
                   const T* __restrict__ v, T* __restrict__ out, int N, int P,
                   int seg_len, int causal, float eps,
                   const float* __restrict__ ws) {
  constexpr int RG = NT / DV;
  constexpr int E = DK / RG;      // S rows per thread (update)
  constexpr int TR = TT / RG;     // tile rows per thread (numerators)
  constexpr int LDK = DK + 1;
  extern __shared__ float sm[];
  float* S = sm;                  // [DK][DV]
  float* z = S + DK * DV;         // [DK]
  float* fq = z + DK;             // [TT][LDK]
  float* fk = fq + TT * LDK;      // [TT][LDK]
  float* vv = fk + TT * LDK;      // [TT][DV]
  float* A = vv + TT * DV;        // [TT][TT+1] masked scores
  float* den = A + TT * (TT + 1); // [TT]

  const long long bh = blockIdx.x;
  const int p = blockIdx.y;
  const int t0 = p * seg_len;
  const int t1 = min(N, t0 + seg_len);
  const int tid = threadIdx.x;
  const int m = tid % DV;
  const int r0 = tid / DV;
  const T* qb = q + bh * N * DK;
  const T* kb = k + bh * N * DK;
  const T* vb = v + bh * N * DV;
  T* ob = out + bh * N * DV;

  const float* st = ws + (bh * P + p) * (long long)(DK * DV + DK);
  for (int i = tid; i < DK * DV + DK; i += NT) S[i] = st[i];  // z follows S
  __syncthreads();

  for (int s = t0; s < t1; s += TT) {
    const int n = min(TT, t1 - s);
    for (int idx = tid; idx < TT * DK; idx += NT) {
      const int t = idx / DK, c = idx % DK;
      const bool in = t < n;
      fq[t * LDK + c] = in ? phi(ld(qb + (long long)(s + t) * DK + c)) : 0.f;
      if (causal) fk[t * LDK + c] = in ? phi(ld(kb + (long long)(s + t) * DK + c)) : 0.f;
    }
    if (causal)
      for (int idx = tid; idx < TT * DV; idx += NT) {
        const int t = idx / DV, c = idx % DV;
        vv[idx] = t < n ? ld(vb + (long long)(s + t) * DV + c) : 0.f;
      }
    __syncthreads();
    if (causal) {
      for (int idx = tid; idx < TT * TT; idx += NT) {
        const int t = idx / TT, j = idx % TT;
        float a = 0.f;
        if (j <= t && t < n) {
#pragma unroll 8
          for (int c = 0; c < DK; ++c) a = fmaf(fq[t * LDK + c], fk[j * LDK + c], a);
        }
        A[t * (TT + 1) + j] = a;
      }
      __syncthreads();
    }
    if (tid < TT) {
      const int t = tid;
      float d = 0.f;
      for (int c = 0; c < DK; ++c) d = fmaf(fq[t * LDK + c], z[c], d);
      if (causal)
        for (int j = 0; j <= t; ++j) d += A[t * (TT + 1) + j];
      den[t] = d + eps;
    }
    float num[TR];
#pragma unroll
    for (int r = 0; r < TR; ++r) {
      const int t = r0 + r * RG;
      float a = 0.f;
#pragma unroll 8
      for (int c = 0; c < DK; ++c) a = fmaf(fq[t * LDK + c], S[c * DV + m], a);
      if (causal)
        for (int j = 0; j <= t; ++j) a = fmaf(A[t * (TT + 1) + j], vv[j * DV + m], a);
      num[r] = a;
    }
    __syncthreads();  // den ready; every read of S for this tile done
#pragma unroll
    for (int r = 0; r < TR; ++r) {
      const int t = r0 + r * RG;
      if (t < n) ob[(long long)(s + t) * DV + m] = from_f32<T>(num[r] / den[t]);
    }
    if (causal) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int c = r0 + e * RG;
        float a = S[c * DV + m];
        for (int t = 0; t < n; ++t) a = fmaf(fk[t * LDK + c], vv[t * DV + m], a);
        S[c * DV + m] = a;
      }
      if (tid < DK) {
        float a = z[tid];
        for (int t = 0; t < n; ++t) a += fk[t * LDK + tid];
        z[tid] = a;
      }
    }
    __syncthreads();
  }
}

template <int DK, int DV, typename T>
cudaError_t launch_state(const FwdArgs& a) {
  dim3 grid(a.BH, a.plan.P);
  simt_state_kernel<DK, DV, T><<<grid, NT, 0, a.stream>>>(
      (const T*)a.k, (const T*)a.v, a.N, a.plan.P, a.plan.seg_len, a.ws_state, a.alpha, a.H);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

template <int DK, int DV, typename T>
cudaError_t launch_output(const FwdArgs& a) {
  constexpr size_t smem = output_smem_bytes<DK, DV>();
  auto kern = simt_output_kernel<DK, DV, T>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid(a.BH, a.plan.P);
  kern<<<grid, NT, smem, a.stream>>>((const T*)a.q, (const T*)a.k, (const T*)a.v,
                                     (T*)a.out, a.N, a.plan.P, a.plan.seg_len,
                                     a.causal, a.eps, a.ws_state);
  err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace

#define LA_PASTE2(a, b) a##b
#define LA_PASTE(a, b) LA_PASTE2(a, b)

cudaError_t LA_PASTE(simt_segment_state_dk, LA_DK)(const FwdArgs& a) {
  const bool bf = a.dtype == LA_BF16;
  switch (a.dv) {
    case 16: return bf ? launch_state<LA_DK, 16, __nv_bfloat16>(a) : launch_state<LA_DK, 16, float>(a);
    case 32: return bf ? launch_state<LA_DK, 32, __nv_bfloat16>(a) : launch_state<LA_DK, 32, float>(a);
    case 64: return bf ? launch_state<LA_DK, 64, __nv_bfloat16>(a) : launch_state<LA_DK, 64, float>(a);
    case 128: return bf ? launch_state<LA_DK, 128, __nv_bfloat16>(a) : launch_state<LA_DK, 128, float>(a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t LA_PASTE(simt_forward_output_dk, LA_DK)(const FwdArgs& a) {
  const bool bf = a.dtype == LA_BF16;
  switch (a.dv) {
    case 16: return bf ? launch_output<LA_DK, 16, __nv_bfloat16>(a) : launch_output<LA_DK, 16, float>(a);
    case 32: return bf ? launch_output<LA_DK, 32, __nv_bfloat16>(a) : launch_output<LA_DK, 32, float>(a);
    case 64: return bf ? launch_output<LA_DK, 64, __nv_bfloat16>(a) : launch_output<LA_DK, 64, float>(a);
    case 128: return bf ? launch_output<LA_DK, 128, __nv_bfloat16>(a) : launch_output<LA_DK, 128, float>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace la
