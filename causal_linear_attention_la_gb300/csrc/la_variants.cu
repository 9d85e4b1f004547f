// State-update variants of the decode path, and the state copy.
//
// Decay gating ("Linear Attention, 곱의 순서를 바꾸면 생기는 일", the paragraph on
// 감쇠 게이팅 after section "요약에는 자리가 모자란다"; the recurrence
// h_t = a h_{t-1} + x_t of "상태공간모델·선형 어텐션", section 3): the whole
// summary (S, z) is multiplied by alpha < 1 before each token is added,
//   S <- alpha S + phi(k) v^T,  z <- alpha z + phi(k),
//   out = phi(q)^T S / (phi(q)^T z + eps).
// Delta rule (the same page, the paragraph on 델타 규칙): read the state with
// the key first and add only the difference to the value,
//   u = S^T k,  S <- S + k (v - u)^T,  out = S^T q,
// with q, k as given (the page works on already-transformed keys; no feature
// map, no normaliser).
//
// Both take T tokens per (b,h) in one CTA with the state in registers, as the
// multi-token decode kernel does: thread (rg, cg) holds rows rg*E .. rg*E+E-1
// and columns 4cg .. 4cg+3; tokens are staged in shared memory in groups.
#include "la_internal.cuh"
#include "la_variants.cuh"

namespace la {

namespace {

template <int DK, int DV>
struct VShape {
  static constexpr int CG = DV / 4;                                // float4 column groups
  static constexpr int NT = (CG * DK) < 256 ? (CG * DK) : 256;    // threads
  static constexpr int RG = NT / CG;                               // row groups
  static constexpr int E = DK / RG;                                // rows per thread
  static constexpr int TG = 16;                                    // tokens per staged group
};

// this thread's E values of a row vector x[rg*E ..]
template <int E>
__device__ __forceinline__ void load_rows(const float* x, float (&r)[E]) {
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 f = *reinterpret_cast<const float4*>(x + e);
      r[e] = f.x; r[e + 1] = f.y; r[e + 2] = f.z; r[e + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) r[e] = x[e];
  }
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(VShape<DK, DV>::NT)
decay_tokens_kernel(float* __restrict__ S, float* __restrict__ z, const T* __restrict__ q,
                    const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ out,
                    const float* __restrict__ alpha, int H, int ntok, float eps) {
  using Sh = VShape<DK, DV>;
  constexpr int NT = Sh::NT, CG = Sh::CG, RG = Sh::RG, E = Sh::E, TG = Sh::TG;
  static_assert(NT % 32 == 0 && E >= 1 && NT >= DK && NT >= DV, "layout");
  __shared__ __align__(16) float fq[TG][DK];
  __shared__ __align__(16) float fk[TG][DK];
  __shared__ __align__(16) float vs[TG][DV];
  __shared__ __align__(16) float part[2][RG][DV];
  __shared__ float wden[2][NT / 32];

  const long long bh = blockIdx.x;
  const int tid = threadIdx.x, cg = tid % CG, rg = tid / CG;
  const float a = alpha[bh % H];
  const T* qb = q + bh * (long long)ntok * DK;
  const T* kb = k + bh * (long long)ntok * DK;
  const T* vb = v + bh * (long long)ntok * DV;
  T* ob = out + bh * (long long)ntok * DV;
  float4* Sb = reinterpret_cast<float4*>(S + bh * (long long)DK * DV);
  float4 s[E];
#pragma unroll
  for (int e = 0; e < E; ++e) s[e] = Sb[(rg * E + e) * CG + cg];
  float zr = tid < DK ? z[bh * DK + tid] : 0.f;
  for (int g0 = 0; g0 < ntok; g0 += TG) {
    const int n = min(TG, ntok - g0);
    __syncthreads();   // the previous group's inputs have been read
    for (int idx = tid; idx < n * DK; idx += NT) {
      fq[idx / DK][idx % DK] = phi(to_f32<T>(qb[(long long)g0 * DK + idx]));
      fk[idx / DK][idx % DK] = phi(to_f32<T>(kb[(long long)g0 * DK + idx]));
    }
    for (int idx = tid; idx < n * DV; idx += NT) vs[idx / DV][idx % DV] = to_f32<T>(vb[(long long)g0 * DV + idx]);
    __syncthreads();
    for (int t = 0; t < n; ++t) {
      const int b = t & 1;
      float zden = 0.f;
      if (tid < DK) {
        zr = fmaf(a, zr, fk[t][tid]);
        zden = fq[t][tid] * zr;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) zden += __shfl_xor_sync(0xffffffffu, zden, o);
      if ((tid & 31) == 0) wden[b][tid >> 5] = zden;
      const float4 vv = *reinterpret_cast<const float4*>(&vs[t][4 * cg]);
      float ka[E], qa[E];
      load_rows<E>(&fk[t][rg * E], ka);
      load_rows<E>(&fq[t][rg * E], qa);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        s[e].x = fmaf(ka[e], vv.x, a * s[e].x);
        s[e].y = fmaf(ka[e], vv.y, a * s[e].y);
        s[e].z = fmaf(ka[e], vv.z, a * s[e].z);
        s[e].w = fmaf(ka[e], vv.w, a * s[e].w);
        acc.x = fmaf(qa[e], s[e].x, acc.x);
        acc.y = fmaf(qa[e], s[e].y, acc.y);
        acc.z = fmaf(qa[e], s[e].z, acc.z);
        acc.w = fmaf(qa[e], s[e].w, acc.w);
      }
      *reinterpret_cast<float4*>(&part[b][rg][4 * cg]) = acc;
      __syncthreads();
      // buffer b is rewritten two tokens later, after the next token's barrier
      if (tid < DV) {
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int r = 0; r < RG; ++r) num += part[b][r][tid];
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) den += wden[b][w];
        ob[(long long)(g0 + t) * DV + tid] = from_f32<T>(num / (den + eps));
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) Sb[(rg * E + e) * CG + cg] = s[e];
  if (tid < DK) z[bh * DK + tid] = zr;
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(VShape<DK, DV>::NT)
delta_tokens_kernel(float* __restrict__ S, const T* __restrict__ q, const T* __restrict__ k,
                    const T* __restrict__ v, T* __restrict__ out, int ntok) {
  using Sh = VShape<DK, DV>;
  constexpr int NT = Sh::NT, CG = Sh::CG, RG = Sh::RG, E = Sh::E, TG = Sh::TG;
  static_assert(NT % 32 == 0 && E >= 1 && NT >= DK && NT >= DV, "layout");
  __shared__ __align__(16) float xq[TG][DK];
  __shared__ __align__(16) float xk[TG][DK];
  __shared__ __align__(16) float vs[TG][DV];
  __shared__ __align__(16) float partk[RG][DV];
  __shared__ __align__(16) float partq[RG][DV];

  const long long bh = blockIdx.x;
  const int tid = threadIdx.x, cg = tid % CG, rg = tid / CG;
  const T* qb = q + bh * (long long)ntok * DK;
  const T* kb = k + bh * (long long)ntok * DK;
  const T* vb = v + bh * (long long)ntok * DV;
  T* ob = out + bh * (long long)ntok * DV;
  float4* Sb = reinterpret_cast<float4*>(S + bh * (long long)DK * DV);
  float4 s[E];
#pragma unroll
  for (int e = 0; e < E; ++e) s[e] = Sb[(rg * E + e) * CG + cg];
  for (int g0 = 0; g0 < ntok; g0 += TG) {
    const int n = min(TG, ntok - g0);
    __syncthreads();   // the previous group's inputs have been read
    for (int idx = tid; idx < n * DK; idx += NT) {
      xq[idx / DK][idx % DK] = to_f32<T>(qb[(long long)g0 * DK + idx]);
      xk[idx / DK][idx % DK] = to_f32<T>(kb[(long long)g0 * DK + idx]);
    }
    for (int idx = tid; idx < n * DV; idx += NT) vs[idx / DV][idx % DV] = to_f32<T>(vb[(long long)g0 * DV + idx]);
    __syncthreads();
    for (int t = 0; t < n; ++t) {
      float ka[E], qa[E];
      load_rows<E>(&xk[t][rg * E], ka);
      load_rows<E>(&xq[t][rg * E], qa);
      // u = S^T k over this thread's rows
      float4 pk = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        pk.x = fmaf(ka[e], s[e].x, pk.x);
        pk.y = fmaf(ka[e], s[e].y, pk.y);
        pk.z = fmaf(ka[e], s[e].z, pk.z);
        pk.w = fmaf(ka[e], s[e].w, pk.w);
      }
      *reinterpret_cast<float4*>(&partk[rg][4 * cg]) = pk;
      __syncthreads();
      // every thread sums u for its own four columns
      float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const float4 p = *reinterpret_cast<const float4*>(&partk[r][4 * cg]);
        u.x += p.x; u.y += p.y; u.z += p.z; u.w += p.w;
      }
      const float4 vv = *reinterpret_cast<const float4*>(&vs[t][4 * cg]);
      const float4 d = make_float4(vv.x - u.x, vv.y - u.y, vv.z - u.z, vv.w - u.w);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        s[e].x = fmaf(ka[e], d.x, s[e].x);
        s[e].y = fmaf(ka[e], d.y, s[e].y);
        s[e].z = fmaf(ka[e], d.z, s[e].z);
        s[e].w = fmaf(ka[e], d.w, s[e].w);
        acc.x = fmaf(qa[e], s[e].x, acc.x);
        acc.y = fmaf(qa[e], s[e].y, acc.y);
        acc.z = fmaf(qa[e], s[e].z, acc.z);
        acc.w = fmaf(qa[e], s[e].w, acc.w);
      }
      *reinterpret_cast<float4*>(&partq[rg][4 * cg]) = acc;
      __syncthreads();
      // partk and partq are rewritten only after the next barrier that every
      // thread reaches after these reads
      if (tid < DV) {
        float num = 0.f;
#pragma unroll
        for (int r = 0; r < RG; ++r) num += partq[r][tid];
        ob[(long long)(g0 + t) * DV + tid] = from_f32<T>(num);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) Sb[(rg * E + e) * CG + cg] = s[e];
}

__global__ void copy_kernel(float4* __restrict__ dst, const float4* __restrict__ src, long long n4) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

template <int DK, int DV, typename T>
cudaError_t launch_decay(const VariantArgs& a) {
  decay_tokens_kernel<DK, DV, T><<<a.BH, VShape<DK, DV>::NT, 0, a.stream>>>(
      a.S, a.z, (const T*)a.q, (const T*)a.k, (const T*)a.v, (T*)a.out, a.alpha, a.H, a.ntok, a.eps);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <int DK, int DV, typename T>
cudaError_t launch_delta(const VariantArgs& a) {
  delta_tokens_kernel<DK, DV, T><<<a.BH, VShape<DK, DV>::NT, 0, a.stream>>>(
      a.S, (const T*)a.q, (const T*)a.k, (const T*)a.v, (T*)a.out, a.ntok);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace

#define LA_VARIANT_SWITCH(FN)                                                         \
  switch (a.dk * 1000 + a.dv) {                                                       \
    LA_VCASE(FN, 16, 16) LA_VCASE(FN, 16, 32) LA_VCASE(FN, 16, 64) LA_VCASE(FN, 16, 128) \
    LA_VCASE(FN, 32, 16) LA_VCASE(FN, 32, 32) LA_VCASE(FN, 32, 64) LA_VCASE(FN, 32, 128) \
    LA_VCASE(FN, 64, 16) LA_VCASE(FN, 64, 32) LA_VCASE(FN, 64, 64) LA_VCASE(FN, 64, 128) \
    LA_VCASE(FN, 128, 16) LA_VCASE(FN, 128, 32) LA_VCASE(FN, 128, 64) LA_VCASE(FN, 128, 128) \
    default: return cudaErrorInvalidValue;                                            \
  }
#define LA_VCASE(FN, DK_, DV_)                                                        \
  case DK_ * 1000 + DV_:                                                              \
    return a.dtype == LA_BF16 ? FN<DK_, DV_, __nv_bfloat16>(a) : FN<DK_, DV_, float>(a);

cudaError_t decode_steps_decay(const VariantArgs& a) { LA_VARIANT_SWITCH(launch_decay) }
cudaError_t decode_steps_delta(const VariantArgs& a) { LA_VARIANT_SWITCH(launch_delta) }

#undef LA_VCASE
#undef LA_VARIANT_SWITCH

cudaError_t copy_floats(float* dst, const float* src, long long n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const long long n4 = n / 4;     // callers pass multiples of 4 floats
  const int threads = 256;
  const long long blocks = (n4 + threads - 1) / threads;
  copy_kernel<<<(int)(blocks < 152 * 8 ? blocks : 152 * 8), threads, 0, stream>>>(
      reinterpret_cast<float4*>(dst), reinterpret_cast<const float4*>(src), n4);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace la
