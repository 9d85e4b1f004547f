// CUDA-core backward kernels (every head size, f32 or bf16), instantiated for
// one key head size LA_DK per translation unit.
//
// Gradients of L = sum(dout * out) by cumulative sums, storing no per-token
// states ("Transformers are RNNs" review, section "그래디언트 계산 — 선형
// 시간·상수 메모리"; the formulas below are derived from the forward
// definition). With g_t = dout_t, D_t = phi(q_t).z_t + eps, o_t = S_t^T phi(q_t)/D_t:
//   a_t = g_t / D_t,  b_t = -(g_t . o_t) / D_t
//   dphi(q_t) = S_t a_t + b_t z_t
//   R_j = sum_{t>=j} phi(q_t) a_t^T,  r_j = sum_{t>=j} b_t phi(q_t)
//   dphi(k_j) = R_j v_j + r_j,  dv_j = R_j^T phi(k_j)
// Tiled form (tile of TT tokens after state S_prev, z_prev; before suffix R_next):
//   W_tj  = phi(q_t).phi(k_j)            for j <= t in the tile
//   dW_tj = a_t . v_j + b_t              for j <= t in the tile
//   dphi(q_t) = sum_j dW_tj phi(k_j) + S_prev a_t + b_t z_prev
//   dphi(k_j) = sum_{t>=j} dW_tj phi(q_t) + R_next v_j + r_next
//   dv_j      = sum_{t>=j} W_tj a_t      + R_next^T phi(k_j)
// Sweep 1 runs forward, writes dq, the per-token scalars D_t, b_t and the
// per-segment reverse sums (dR, dr); after a reverse segment scan, sweep 2
// runs backward through each segment and writes dk, dv.
// Decay gating (alpha: per-head factors, else null; causal): S_t = alpha
// S_{t-1} + phi(k_t) v_t^T and z likewise ("Linear Attention, 곱의 순서를
// 바꾸면 생기는 일", paragraph on 감쇠 게이팅), and the reverse sums decay the
// same way, R_j = phi(q_j) a_j^T + alpha R_{j+1}. In a tile the pair (t, j)
// carries alpha^(t-j), the tile's starting state alpha^(t+1) at row t, the
// suffix after the tile alpha^(n-j) at key j; records are decayed to their
// segment's last token (forward) or first token (reverse) and the segment
// scan decays across segments.
#include "la_internal.cuh"

#ifndef LA_DK
#error "define LA_DK before including this file"
#endif

namespace la {

namespace {

constexpr int NT = 256;
constexpr int TT = 32;

template <typename T>
__device__ __forceinline__ float ld(const T* p) { return to_f32<T>(*p); }

// init + sum_{i < n} x[i sx] y[i sy] with four independent partial sums, so
// that a thread's FMAs do not wait on each other
__device__ __forceinline__ float dot4(const float* x, int sx, const float* y, int sy, int n, float init = 0.f) {
  float a0 = init, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  int i = 0;
  for (; i + 4 <= n; i += 4) {
    a0 = fmaf(x[i * sx], y[i * sy], a0);
    a1 = fmaf(x[(i + 1) * sx], y[(i + 1) * sy], a1);
    a2 = fmaf(x[(i + 2) * sx], y[(i + 2) * sy], a2);
    a3 = fmaf(x[(i + 3) * sx], y[(i + 3) * sy], a3);
  }
  for (; i < n; ++i) a0 = fmaf(x[i * sx], y[i * sy], a0);
  return (a0 + a1) + (a2 + a3);
}

template <int DK, int DV>
constexpr size_t sweep1_smem_floats() {
  // S, z, fq, fk, vv, gg, aa, oo(stage), W, dW, den, bsc
  return (size_t)DK * DV + DK + 2 * TT * (DK + 1) + 3 * TT * (DV + 1) +
         (size_t)TT * ((DK > DV ? DK : DV) + 1) + 2 * TT * (TT + 1) + 2 * TT;
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(NT)
simt_bwd_sweep1(const T* __restrict__ q, const T* __restrict__ k,
                const T* __restrict__ v, const T* __restrict__ g,
                T* __restrict__ dq, int N, int P, int seg_len, int causal,
                float eps, const float* __restrict__ ws_state,
                float* __restrict__ ws_rev, float* __restrict__ ws_tok,
                const float* __restrict__ alpha, int H) {
  constexpr int LDK = DK + 1, LDV = DV + 1;
  constexpr int LST = (DK > DV ? DK : DV) + 1;
  constexpr int RG = NT / DV;     // (c, m) layout: m = tid % DV
  constexpr int E = DK / RG;
  constexpr int TR = TT / RG;     // (t, m) layout
  constexpr int CG = NT / TT;     // (t, c) layout: t = tid % TT
  constexpr int EC = DK / CG;
  extern __shared__ float sm[];
  float* S = sm;
  float* z = S + DK * DV;
  float* fq = z + DK;
  float* fk = fq + TT * LDK;
  float* vv = fk + TT * LDK;
  float* gg = vv + TT * LDV;
  float* aa = gg + TT * LDV;
  float* stg = aa + TT * LDV;     // o_t, then dq staging
  float* W = stg + TT * LST;
  float* dW = W + TT * (TT + 1);
  float* den = dW + TT * (TT + 1);
  float* bsc = den + TT;

  const long long bh = blockIdx.x;
  const int p = blockIdx.y;
  const int t0 = p * seg_len;
  const int t1 = min(N, t0 + seg_len);
  const int tid = threadIdx.x;
  const T* qb = q + bh * N * DK;
  const T* kb = k + bh * N * DK;
  const T* vb = v + bh * N * DV;
  const T* gb = g + bh * N * DV;
  T* dqb = dq + bh * N * DK;
  float* tok = ws_tok + bh * (long long)N * 2;

  const float* st = ws_state + (bh * P + p) * (long long)(DK * DV + DK);
  for (int i = tid; i < DK * DV + DK; i += NT) S[i] = st[i];

  const int m = tid % DV, c0 = tid / DV;
  float racc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) racc[e] = 0.f;
  float rz = 0.f;
  const float log2a = alpha != nullptr ? log2f(alpha[bh % H]) : 0.f;
  const bool decay = alpha != nullptr;
  // alpha^e (1 without decay: no exponential in the inner loops)
  auto dec = [&](int e) { return decay ? exp2f((float)e * log2a) : 1.f; };
  __syncthreads();

  for (int s = t0; s < t1; s += TT) {
    const int n = min(TT, t1 - s);
    for (int idx = tid; idx < TT * DK; idx += NT) {
      const int t = idx / DK, c = idx % DK;
      const bool in = t < n;
      fq[t * LDK + c] = in ? phi(ld(qb + (long long)(s + t) * DK + c)) : 0.f;
      fk[t * LDK + c] = in ? phi(ld(kb + (long long)(s + t) * DK + c)) : 0.f;
    }
    for (int idx = tid; idx < TT * DV; idx += NT) {
      const int t = idx / DV, c = idx % DV;
      const bool in = t < n;
      vv[t * LDV + c] = in ? ld(vb + (long long)(s + t) * DV + c) : 0.f;
      gg[t * LDV + c] = in ? ld(gb + (long long)(s + t) * DV + c) : 0.f;
    }
    __syncthreads();
    if (causal) {
      for (int idx = tid; idx < TT * TT; idx += NT) {
        const int t = idx / TT, j = idx % TT;
        float a = 0.f;
        if (j <= t && t < n) a = dot4(fq + t * LDK, 1, fk + j * LDK, 1, DK) * dec(t - j);
        W[t * (TT + 1) + j] = a;
      }
      __syncthreads();
    }
    if (tid < TT) {
      const int t = tid;
      float d = dot4(fq + t * LDK, 1, z, 1, DK) * dec(t + 1);
      if (causal)
        for (int j = 0; j <= t; ++j) d += W[t * (TT + 1) + j];
      den[t] = t < n ? d + eps : 1.f;  // padding rows stay finite when eps = 0
    }
    float num[TR];
    for (int r = 0; r < TR; ++r) {
      const int t = tid / DV + r * RG;
      float a = dot4(fq + t * LDK, 1, S + m, DV, DK) * dec(t + 1);
      if (causal) a = dot4(W + t * (TT + 1), 1, vv + m, LDV, t + 1, a);
      num[r] = a;
    }
    __syncthreads();
    for (int r = 0; r < TR; ++r) {
      const int t = tid / DV + r * RG;
      const float inv = 1.f / den[t];
      stg[t * LST + m] = num[r] * inv;        // o_t
      aa[t * LDV + m] = gg[t * LDV + m] * inv;  // a_t
    }
    __syncthreads();
    if (tid < TT) {
      const int t = tid;
      const float beta = dot4(gg + t * LDV, 1, stg + t * LST, 1, DV);
      const float b = -beta / den[t];
      bsc[t] = t < n ? b : 0.f;
      if (t < n) {
        tok[(long long)(s + t) * 2 + 0] = den[t];
        tok[(long long)(s + t) * 2 + 1] = b;
      }
    }
    __syncthreads();
    if (causal) {
      for (int idx = tid; idx < TT * TT; idx += NT) {
        const int t = idx / TT, j = idx % TT;
        float a = 0.f;
        if (j <= t && t < n) a = (dot4(aa + t * LDV, 1, vv + j * LDV, 1, DV) + bsc[t]) * dec(t - j);
        dW[t * (TT + 1) + j] = a;
      }
      __syncthreads();
    }
    // dphi(q) in (t, c) layout, staged for a coalesced store
    {
      const int t = tid % TT;
      for (int e = 0; e < EC; ++e) {
        const int c = tid / TT + e * CG;
        float a = dot4(aa + t * LDV, 1, S + c * DV, 1, DV, bsc[t] * z[c]) * dec(t + 1);
        if (causal) a = dot4(dW + t * (TT + 1), 1, fk + c, LDK, t + 1, a);
        stg[t * LST + c] = a * phi_prime_from_phi(fq[t * LDK + c]);
      }
    }
    __syncthreads();
    for (int idx = tid; idx < TT * DK; idx += NT) {
      const int t = idx / DK, c = idx % DK;
      if (t < n) dqb[(long long)(s + t) * DK + c] = from_f32<T>(stg[t * LST + c]);
    }
    // segment reverse sums dR += phi(q)^T a, dr += sum_t b_t phi(q_t)
    // (decayed to the segment's first token)
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = c0 + e * RG;
      float a = racc[e];
      if (decay)
        for (int t = 0; t < n; ++t) a = fmaf(fq[t * LDK + c] * dec(s + t - t0), aa[t * LDV + m], a);
      else
        a = dot4(fq + c, LDK, aa + m, LDV, n, a);
      racc[e] = a;
    }
    if (tid < DK) {
      if (decay)
        for (int t = 0; t < n; ++t) rz = fmaf(bsc[t] * dec(s + t - t0), fq[t * LDK + tid], rz);
      else
        rz = dot4(bsc, 1, fq + tid, LDK, n, rz);
    }
    if (causal) {
      // the state after the tile: alpha^n S + sum_j alpha^(n-1-j) phi(k_j) v_j^T
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int c = c0 + e * RG;
        float a = S[c * DV + m] * dec(n);
        if (decay)
          for (int t = 0; t < n; ++t) a = fmaf(fk[t * LDK + c] * dec(n - 1 - t), vv[t * LDV + m], a);
        else
          a = dot4(fk + c, LDK, vv + m, LDV, n, a);
        S[c * DV + m] = a;
      }
      if (tid < DK) {
        float a = z[tid] * dec(n);
        for (int t = 0; t < n; ++t) a = fmaf(fk[t * LDK + tid], dec(n - 1 - t), a);
        z[tid] = a;
      }
    }
    __syncthreads();
  }
  float* o = ws_rev + (bh * P + p) * (long long)(DK * DV + DK);
#pragma unroll
  for (int e = 0; e < E; ++e) o[(c0 + e * RG) * DV + m] = racc[e];
  if (tid < DK) o[DK * DV + tid] = rz;
}

template <int DK, int DV>
constexpr size_t sweep2_smem_floats() {
  // R, r, fq, fk, vv, aa, W, dW, bsc, den, dk stage, dv stage
  return (size_t)DK * DV + DK + 2 * TT * (DK + 1) + 2 * TT * (DV + 1) +
         2 * TT * (TT + 1) + 2 * TT + TT * (DK + 1) + TT * (DV + 1);
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(NT)
simt_bwd_sweep2(const T* __restrict__ q, const T* __restrict__ k,
                const T* __restrict__ v, const T* __restrict__ g,
                T* __restrict__ dk_, T* __restrict__ dv_, int N, int P,
                int seg_len, int causal, const float* __restrict__ ws_rev,
                const float* __restrict__ ws_tok, const float* __restrict__ alpha, int H) {
  constexpr int LDK = DK + 1, LDV = DV + 1;
  constexpr int RG = NT / DV;
  constexpr int E = DK / RG;
  constexpr int CG = NT / TT;
  constexpr int EC = DK / CG;
  constexpr int EM = DV / CG;
  extern __shared__ float sm[];
  float* R = sm;
  float* r = R + DK * DV;
  float* fq = r + DK;
  float* fk = fq + TT * LDK;
  float* vv = fk + TT * LDK;
  float* aa = vv + TT * LDV;
  float* W = aa + TT * LDV;
  float* dW = W + TT * (TT + 1);
  float* bsc = dW + TT * (TT + 1);
  float* den = bsc + TT;
  float* sdk = den + TT;
  float* sdv = sdk + TT * LDK;

  const long long bh = blockIdx.x;
  const int p = blockIdx.y;
  const int t0 = p * seg_len;
  const int t1 = min(N, t0 + seg_len);
  const int tid = threadIdx.x;
  const T* qb = q + bh * N * DK;
  const T* kb = k + bh * N * DK;
  const T* vb = v + bh * N * DV;
  const T* gb = g + bh * N * DV;
  T* dkb = dk_ + bh * N * DK;
  T* dvb = dv_ + bh * N * DV;
  const float* tok = ws_tok + bh * (long long)N * 2;

  const float* st = ws_rev + (bh * P + p) * (long long)(DK * DV + DK);
  for (int i = tid; i < DK * DV + DK; i += NT) R[i] = st[i];
  const int m = tid % DV, c0 = tid / DV;
  const float log2a = alpha != nullptr ? log2f(alpha[bh % H]) : 0.f;
  const bool decay = alpha != nullptr;
  // alpha^e (1 without decay: no exponential in the inner loops)
  auto dec = [&](int e) { return decay ? exp2f((float)e * log2a) : 1.f; };
  __syncthreads();

  const int ntiles = (t1 - t0 + TT - 1) / TT;
  for (int it = ntiles - 1; it >= 0; --it) {
    const int s = t0 + it * TT;
    const int n = min(TT, t1 - s);
    if (tid < TT) {
      den[tid] = tid < n ? tok[(long long)(s + tid) * 2 + 0] : 1.f;
      bsc[tid] = tid < n ? tok[(long long)(s + tid) * 2 + 1] : 0.f;
    }
    for (int idx = tid; idx < TT * DK; idx += NT) {
      const int t = idx / DK, c = idx % DK;
      const bool in = t < n;
      fq[t * LDK + c] = in ? phi(ld(qb + (long long)(s + t) * DK + c)) : 0.f;
      fk[t * LDK + c] = in ? phi(ld(kb + (long long)(s + t) * DK + c)) : 0.f;
    }
    __syncthreads();  // den visible
    for (int idx = tid; idx < TT * DV; idx += NT) {
      const int t = idx / DV, c = idx % DV;
      const bool in = t < n;
      vv[t * LDV + c] = in ? ld(vb + (long long)(s + t) * DV + c) : 0.f;
      aa[t * LDV + c] = in ? ld(gb + (long long)(s + t) * DV + c) / den[t] : 0.f;
    }
    __syncthreads();
    if (causal) {
      for (int idx = tid; idx < TT * TT; idx += NT) {
        const int t = idx / TT, j = idx % TT;
        float w = 0.f, dw = 0.f;
        if (j <= t && t < n) {
          w = dot4(fq + t * LDK, 1, fk + j * LDK, 1, DK);
          dw = dot4(aa + t * LDV, 1, vv + j * LDV, 1, DV);
          const float f = dec(t - j);
          w *= f;
          dw = (dw + bsc[t]) * f;
        }
        W[t * (TT + 1) + j] = w;
        dW[t * (TT + 1) + j] = dw;
      }
      __syncthreads();
    }
    {
      const int j = tid % TT;
      for (int e = 0; e < EC; ++e) {
        const int c = tid / TT + e * CG;
        float a = dot4(R + c * DV, 1, vv + j * LDV, 1, DV, r[c]);
        a *= dec(n - j);    // the suffix after the tile, seen from key j
        if (causal) a = dot4(dW + j * (TT + 1) + j, TT + 1, fq + j * LDK + c, LDK, TT - j, a);
        sdk[j * LDK + c] = a * phi_prime_from_phi(fk[j * LDK + c]);
      }
      for (int e = 0; e < EM; ++e) {
        const int mm = tid / TT + e * CG;
        float a = dot4(R + mm, DV, fk + j * LDK, 1, DK) * dec(n - j);
        if (causal) a = dot4(W + j * (TT + 1) + j, TT + 1, aa + j * LDV + mm, LDV, TT - j, a);
        sdv[j * LDV + mm] = a;
      }
    }
    __syncthreads();  // all reads of R for this tile done
    for (int idx = tid; idx < TT * DK; idx += NT) {
      const int t = idx / DK, c = idx % DK;
      if (t < n) dkb[(long long)(s + t) * DK + c] = from_f32<T>(sdk[t * LDK + c]);
    }
    for (int idx = tid; idx < TT * DV; idx += NT) {
      const int t = idx / DV, c = idx % DV;
      if (t < n) dvb[(long long)(s + t) * DV + c] = from_f32<T>(sdv[t * LDV + c]);
    }
    if (causal) {
#pragma unroll
      // the suffix at the tile's first token: alpha^n R + sum_t alpha^t phi(q_t) a_t^T
      for (int e = 0; e < E; ++e) {
        const int c = c0 + e * RG;
        float a = R[c * DV + m] * dec(n);
        if (decay)
          for (int t = 0; t < n; ++t) a = fmaf(fq[t * LDK + c] * dec(t), aa[t * LDV + m], a);
        else
          a = dot4(fq + c, LDK, aa + m, LDV, n, a);
        R[c * DV + m] = a;
      }
      if (tid < DK) {
        float a = r[tid] * dec(n);
        if (decay)
          for (int t = 0; t < n; ++t) a = fmaf(bsc[t] * dec(t), fq[t * LDK + tid], a);
        else
          a = dot4(bsc, 1, fq + tid, LDK, n, a);
        r[tid] = a;
      }
    }
    __syncthreads();
  }
}

template <int DK, int DV, typename T>
cudaError_t launch_bwd(const BwdArgs& a) {
  FwdArgs f{};
  f.q = a.q; f.k = a.k; f.v = a.v; f.out = nullptr;
  f.BH = a.BH; f.N = a.N; f.dk = a.dk; f.dv = a.dv; f.causal = a.causal;
  f.eps = a.eps; f.dtype = a.dtype; f.ws_state = a.ws_state; f.plan = a.plan;
  f.stream = a.stream;
  f.alpha = a.alpha; f.H = a.H;
  const long long words = state_words(DK, DV);
  prof_begin(LA_SPAN_BWD_STATE, a.stream);
  cudaError_t err = simt_segment_state(f);
  if (err == cudaSuccess)
    err = segment_scan(a.ws_state, a.BH, a.plan.P, words,
                       a.causal ? SCAN_EXCLUSIVE_FWD : SCAN_TOTAL, nullptr,
                       nullptr, DK, DV, a.stream, a.alpha, a.H, a.plan.seg_len, a.N);
  prof_end(LA_SPAN_BWD_STATE, a.stream);
  if (err != cudaSuccess) return err;

  dim3 grid(a.BH, a.plan.P);
  constexpr size_t smem1 = sizeof(float) * sweep1_smem_floats<DK, DV>();
  auto k1 = simt_bwd_sweep1<DK, DV, T>;
  err = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
  if (err != cudaSuccess) return err;
  prof_begin(LA_SPAN_BWD_SWEEP1, a.stream);
  k1<<<grid, NT, smem1, a.stream>>>((const T*)a.q, (const T*)a.k, (const T*)a.v,
                                    (const T*)a.dout, (T*)a.dq, a.N, a.plan.P,
                                    a.plan.seg_len, a.causal, a.eps, a.ws_state,
                                    a.ws_rev, a.ws_tok, a.alpha, a.H);
  prof_end(LA_SPAN_BWD_SWEEP1, a.stream);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  note_launch();
  prof_begin(LA_SPAN_BWD_SCAN, a.stream);
  err = segment_scan(a.ws_rev, a.BH, a.plan.P, words,
                     a.causal ? SCAN_EXCLUSIVE_REV : SCAN_TOTAL, nullptr,
                     nullptr, DK, DV, a.stream, a.alpha, a.H, a.plan.seg_len, a.N);
  prof_end(LA_SPAN_BWD_SCAN, a.stream);
  if (err != cudaSuccess) return err;
  constexpr size_t smem2 = sizeof(float) * sweep2_smem_floats<DK, DV>();
  auto k2 = simt_bwd_sweep2<DK, DV, T>;
  err = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
  if (err != cudaSuccess) return err;
  prof_begin(LA_SPAN_BWD_SWEEP2, a.stream);
  k2<<<grid, NT, smem2, a.stream>>>((const T*)a.q, (const T*)a.k, (const T*)a.v,
                                    (const T*)a.dout, (T*)a.dk_, (T*)a.dv_, a.N,
                                    a.plan.P, a.plan.seg_len, a.causal,
                                    a.ws_rev, a.ws_tok, a.alpha, a.H);
  prof_end(LA_SPAN_BWD_SWEEP2, a.stream);
  err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace

#define LA_PASTE2(a, b) a##b
#define LA_PASTE(a, b) LA_PASTE2(a, b)

cudaError_t LA_PASTE(simt_backward_dk, LA_DK)(const BwdArgs& a) {
  const bool bf = a.dtype == LA_BF16;
  switch (a.dv) {
    case 16: return bf ? launch_bwd<LA_DK, 16, __nv_bfloat16>(a) : launch_bwd<LA_DK, 16, float>(a);
    case 32: return bf ? launch_bwd<LA_DK, 32, __nv_bfloat16>(a) : launch_bwd<LA_DK, 32, float>(a);
    case 64: return bf ? launch_bwd<LA_DK, 64, __nv_bfloat16>(a) : launch_bwd<LA_DK, 64, float>(a);
    case 128: return bf ? launch_bwd<LA_DK, 128, __nv_bfloat16>(a) : launch_bwd<LA_DK, 128, float>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace la
