// Decode: one recurrent step per (batch, head), in place on the fp32 state.
//
//   S <- S + phi(k) v^T,  z <- z + phi(k),  out = phi(q)^T S / (phi(q)^T z + eps)
//
// ("Linear Attention: KV를 고정 크기 상태에 누적하기", section "상태 갱신과 읽기를
// 식으로 정리하기"; the step reads the state that already holds the token.)
//
// Memory-bound: each (b,h) reads and writes its dk x dv fp32 state once
// (64 KiB each way at dk = dv = 128). One CTA per (b,h). Each thread owns one
// float4 column group and every RG-th row, so a warp touches whole 512-byte
// rows (coalesced 16-byte accesses), all E loads of a thread are independent
// and in flight together, and the read of the updated row is fused into the
// same pass. phi(q)^T S partials are reduced across row groups in shared
// memory; phi(q)^T z by warp shuffles.
#include "la_internal.cuh"

namespace la {

namespace {

template <int DK, int DV>
struct DecodeShape {
  static constexpr int CG = DV / 4;                                // float4 column groups
  static constexpr int NT = (CG * DK) < 256 ? (CG * DK) : 256;    // threads
  static constexpr int RG = NT / CG;                               // row groups
  static constexpr int E = DK / RG;                                // rows per thread
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(DecodeShape<DK, DV>::NT)
decode_kernel(float* __restrict__ S, float* __restrict__ z,
              const T* __restrict__ q, const T* __restrict__ k,
              const T* __restrict__ v, T* __restrict__ out, float eps) {
  using Sh = DecodeShape<DK, DV>;
  constexpr int NT = Sh::NT, CG = Sh::CG, RG = Sh::RG, E = Sh::E;
  static_assert(NT % 32 == 0 && E >= 1, "decode layout");
  __shared__ __align__(16) float fq[DK];
  __shared__ __align__(16) float fk[DK];
  __shared__ __align__(16) float vs[DV];
  __shared__ __align__(16) float part[RG][DV];
  __shared__ float wden[NT / 32];

  const long long bh = blockIdx.x;
  const int tid = threadIdx.x;
  float zden = 0.f;
  if (tid < DK) {
    const float pk = phi(to_f32<T>(k[bh * DK + tid]));
    const float pq = phi(to_f32<T>(q[bh * DK + tid]));
    fk[tid] = pk;
    fq[tid] = pq;
    const float zn = z[bh * DK + tid] + pk;
    z[bh * DK + tid] = zn;
    zden = pq * zn;
  }
  if (tid < DV) vs[tid] = to_f32<T>(v[bh * DV + tid]);
  // phi(q)^T z: warp shuffle, then across warps
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) zden += __shfl_xor_sync(0xffffffffu, zden, o);
  if ((tid & 31) == 0) wden[tid >> 5] = zden;
  __syncthreads();

  const int cg = tid % CG;
  const int rg = tid / CG;
  const float4 vv = *reinterpret_cast<const float4*>(&vs[4 * cg]);
  float4* Sb = reinterpret_cast<float4*>(S + bh * (long long)DK * DV);
  float4 s[E];
#pragma unroll
  for (int e = 0; e < E; ++e) s[e] = Sb[(rg + e * RG) * CG + cg];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int row = rg + e * RG;
    const float a = fk[row], b = fq[row];
    float4 x = s[e];
    x.x = fmaf(a, vv.x, x.x);
    x.y = fmaf(a, vv.y, x.y);
    x.z = fmaf(a, vv.z, x.z);
    x.w = fmaf(a, vv.w, x.w);
    Sb[row * CG + cg] = x;
    acc.x = fmaf(b, x.x, acc.x);
    acc.y = fmaf(b, x.y, acc.y);
    acc.z = fmaf(b, x.z, acc.z);
    acc.w = fmaf(b, x.w, acc.w);
  }
  *reinterpret_cast<float4*>(&part[rg][4 * cg]) = acc;
  __syncthreads();
  if (tid < DV) {
    float num = 0.f;
#pragma unroll
    for (int r = 0; r < RG; ++r) num += part[r][tid];
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) den += wden[w];
    out[bh * DV + tid] = from_f32<T>(num / (den + eps));
  }
}

// T consecutive tokens of one (b,h) per CTA: the state stays in registers for
// all of them (read and written once per call instead of once per token);
// each token is the step above. Tokens are taken in groups of TG: the group's
// phi(q), phi(k) and v are staged in shared memory by all threads at once
// (one load latency per group), then the group's steps run with one barrier
// each, their partial sums alternating between two buffers.
template <int DK, int DV, typename T>
__global__ void __launch_bounds__(DecodeShape<DK, DV>::NT)
decode_tokens_kernel(float* __restrict__ S, float* __restrict__ z,
                     const T* __restrict__ q, const T* __restrict__ k,
                     const T* __restrict__ v, T* __restrict__ out, int ntok, float eps) {
  using Sh = DecodeShape<DK, DV>;
  constexpr int NT = Sh::NT, CG = Sh::CG, RG = Sh::RG, E = Sh::E;
  constexpr int TG = 16;
  static_assert(NT % 32 == 0 && E >= 1 && NT >= DK && NT >= DV, "decode layout");
  __shared__ __align__(16) float fq[TG][DK];
  __shared__ __align__(16) float fk[TG][DK];
  __shared__ __align__(16) float vs[TG][DV];
  __shared__ __align__(16) float part[2][RG][DV];
  __shared__ float wden[2][NT / 32];

  const long long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int cg = tid % CG;
  const int rg = tid / CG;
  const T* qb = q + bh * (long long)ntok * DK;
  const T* kb = k + bh * (long long)ntok * DK;
  const T* vb = v + bh * (long long)ntok * DV;
  T* ob = out + bh * (long long)ntok * DV;

  // this thread's rows rg*E .. rg*E+E-1 (contiguous, so their phi values are
  // read as vectors), column group cg; a warp still reads whole state rows
  float4* Sb = reinterpret_cast<float4*>(S + bh * (long long)DK * DV);
  float4 s[E];
#pragma unroll
  for (int e = 0; e < E; ++e) s[e] = Sb[(rg * E + e) * CG + cg];
  float zr = tid < DK ? z[bh * DK + tid] : 0.f;       // z[tid], kept by thread tid
  for (int g0 = 0; g0 < ntok; g0 += TG) {
    const int n = min(TG, ntok - g0);
    // the previous group's inputs have been read by every thread
    __syncthreads();
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
        zr += fk[t][tid];
        zden = fq[t][tid] * zr;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) zden += __shfl_xor_sync(0xffffffffu, zden, o);
      if ((tid & 31) == 0) wden[b][tid >> 5] = zden;
      const float4 vv = *reinterpret_cast<const float4*>(&vs[t][4 * cg]);
      float ka[E], qa[E];
      if constexpr (E % 4 == 0) {
#pragma unroll
        for (int e = 0; e < E; e += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(&fk[t][rg * E + e]);
          const float4 q4 = *reinterpret_cast<const float4*>(&fq[t][rg * E + e]);
          ka[e] = k4.x; ka[e + 1] = k4.y; ka[e + 2] = k4.z; ka[e + 3] = k4.w;
          qa[e] = q4.x; qa[e + 1] = q4.y; qa[e + 2] = q4.z; qa[e + 3] = q4.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) { ka[e] = fk[t][rg * E + e]; qa[e] = fq[t][rg * E + e]; }
      }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float a = ka[e], c = qa[e];
        s[e].x = fmaf(a, vv.x, s[e].x);
        s[e].y = fmaf(a, vv.y, s[e].y);
        s[e].z = fmaf(a, vv.z, s[e].z);
        s[e].w = fmaf(a, vv.w, s[e].w);
        acc.x = fmaf(c, s[e].x, acc.x);
        acc.y = fmaf(c, s[e].y, acc.y);
        acc.z = fmaf(c, s[e].z, acc.z);
        acc.w = fmaf(c, s[e].w, acc.w);
      }
      *reinterpret_cast<float4*>(&part[b][rg][4 * cg]) = acc;
      __syncthreads();
      // buffer b is written again two steps later, after the next step's
      // barrier, which every thread reaches only after this read
      if (tid < DV) {
        float num = 0.f;
#pragma unroll
        for (int r = 0; r < RG; ++r) num += part[b][r][tid];
        float den = 0.f;
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
cudaError_t launch(const DecodeArgs& a) {
  if (a.ntok == 1)
    decode_kernel<DK, DV, T><<<a.BH, DecodeShape<DK, DV>::NT, 0, a.stream>>>(
        a.S, a.z, (const T*)a.q, (const T*)a.k, (const T*)a.v, (T*)a.out, a.eps);
  else
    decode_tokens_kernel<DK, DV, T><<<a.BH, DecodeShape<DK, DV>::NT, 0, a.stream>>>(
        a.S, a.z, (const T*)a.q, (const T*)a.k, (const T*)a.v, (T*)a.out, a.ntok, a.eps);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace

cudaError_t decode_step(const DecodeArgs& a) {
#define LA_CASE(DK_, DV_)                                                  \
  case DK_ * 1000 + DV_:                                                   \
    return a.dtype == LA_BF16 ? launch<DK_, DV_, __nv_bfloat16>(a)         \
                              : launch<DK_, DV_, float>(a);
  switch (a.dk * 1000 + a.dv) {
    LA_CASE(16, 16) LA_CASE(16, 32) LA_CASE(16, 64) LA_CASE(16, 128)
    LA_CASE(32, 16) LA_CASE(32, 32) LA_CASE(32, 64) LA_CASE(32, 128)
    LA_CASE(64, 16) LA_CASE(64, 32) LA_CASE(64, 64) LA_CASE(64, 128)
    LA_CASE(128, 16) LA_CASE(128, 32) LA_CASE(128, 64) LA_CASE(128, 128)
    default: return cudaErrorInvalidValue;
  }
#undef LA_CASE
}

}  // namespace la
