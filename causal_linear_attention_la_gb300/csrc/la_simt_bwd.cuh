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
#include <type_traits>

#include "la_internal.cuh"

#ifndef LA_DK
#error "define LA_DK before including this file"
#endif

namespace la {

// dk = dv = 128 without decay: the register-tiled sweeps (their own
// translation unit, la_simt_bwd_t128.cu)
cudaError_t simt_backward_tiled128(const BwdArgs& a);

namespace {

constexpr int NT = 256;
constexpr int TT = 32;

template <typename T>
__device__ __forceinline__ float ld(const T* p) { return to_f32<T>(*p); }

#ifndef LA_TILED128_ONLY
template <int DK, int DV>
constexpr size_t sweep1_smem_floats() {
  // S, z, fq, fk, vv, gg, aa, oo(stage), W, dW, den, bsc, the tile's decay weights
  return (size_t)DK * DV + DK + 2 * TT * (DK + 1) + 3 * TT * (DV + 1) +
         (size_t)TT * ((DK > DV ? DK : DV) + 1) + 2 * TT * (TT + 1) + 2 * TT + 2 * TT;
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
  float* wr = bsc + TT;           // alpha^(token - segment start) of the tile's tokens
  float* wk = wr + TT;            // alpha^(n - 1 - t)

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
  // alpha^e (1 without decay); the innermost loops read per-tile tables instead
  auto dec = [&](int e) { return exp2f((float)e * log2a); };
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
    if (tid < TT) {
      wr[tid] = dec(s + tid - t0);
      wk[tid] = dec(n - 1 - tid);
    }
    __syncthreads();
    if (causal) {
      for (int idx = tid; idx < TT * TT; idx += NT) {
        const int t = idx / TT, j = idx % TT;
        float a = 0.f;
        if (j <= t && t < n) {
          for (int c = 0; c < DK; ++c) a = fmaf(fq[t * LDK + c], fk[j * LDK + c], a);
          a *= dec(t - j);
        }
        W[t * (TT + 1) + j] = a;
      }
      __syncthreads();
    }
    if (tid < TT) {
      const int t = tid;
      float d = 0.f;
      for (int c = 0; c < DK; ++c) d = fmaf(fq[t * LDK + c], z[c], d);
      d *= dec(t + 1);
      if (causal)
        for (int j = 0; j <= t; ++j) d += W[t * (TT + 1) + j];
      den[t] = t < n ? d + eps : 1.f;  // padding rows stay finite when eps = 0
    }
    float num[TR];
    for (int r = 0; r < TR; ++r) {
      const int t = tid / DV + r * RG;
      float a = 0.f;
      for (int c = 0; c < DK; ++c) a = fmaf(fq[t * LDK + c], S[c * DV + m], a);
      a *= dec(t + 1);
      if (causal)
        for (int j = 0; j <= t; ++j) a = fmaf(W[t * (TT + 1) + j], vv[j * LDV + m], a);
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
      float beta = 0.f;
      for (int mm = 0; mm < DV; ++mm) beta = fmaf(gg[t * LDV + mm], stg[t * LST + mm], beta);
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
        if (j <= t && t < n) {
          for (int mm = 0; mm < DV; ++mm) a = fmaf(aa[t * LDV + mm], vv[j * LDV + mm], a);
          a = (a + bsc[t]) * dec(t - j);
        }
        dW[t * (TT + 1) + j] = a;
      }
      __syncthreads();
    }
    // dphi(q) in (t, c) layout, staged for a coalesced store
    {
      const int t = tid % TT;
      for (int e = 0; e < EC; ++e) {
        const int c = tid / TT + e * CG;
        float a = bsc[t] * z[c];
        for (int mm = 0; mm < DV; ++mm) a = fmaf(aa[t * LDV + mm], S[c * DV + mm], a);
        a *= dec(t + 1);
        if (causal)
          for (int j = 0; j <= t; ++j) a = fmaf(dW[t * (TT + 1) + j], fk[j * LDK + c], a);
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
      for (int t = 0; t < n; ++t) a = fmaf(fq[t * LDK + c] * wr[t], aa[t * LDV + m], a);
      racc[e] = a;
    }
    if (tid < DK)
      for (int t = 0; t < n; ++t) rz = fmaf(bsc[t] * wr[t], fq[t * LDK + tid], rz);
    if (causal) {
      // the state after the tile: alpha^n S + sum_j alpha^(n-1-j) phi(k_j) v_j^T
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int c = c0 + e * RG;
        float a = S[c * DV + m] * dec(n);
        for (int t = 0; t < n; ++t) a = fmaf(fk[t * LDK + c] * wk[t], vv[t * LDV + m], a);
        S[c * DV + m] = a;
      }
      if (tid < DK) {
        float a = z[tid] * dec(n);
        for (int t = 0; t < n; ++t) a = fmaf(fk[t * LDK + tid], wk[t], a);
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
  // R, r, fq, fk, vv, aa, W, dW, bsc, den, dk stage, dv stage, the tile's decay weights
  return (size_t)DK * DV + DK + 2 * TT * (DK + 1) + 2 * TT * (DV + 1) +
         2 * TT * (TT + 1) + 2 * TT + TT * (DK + 1) + TT * (DV + 1) + TT;
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
  float* wt = sdv + TT * LDV;     // alpha^t of the tile's tokens

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
  // alpha^e (1 without decay); the innermost loops read per-tile tables instead
  auto dec = [&](int e) { return exp2f((float)e * log2a); };
  __syncthreads();

  const int ntiles = (t1 - t0 + TT - 1) / TT;
  for (int it = ntiles - 1; it >= 0; --it) {
    const int s = t0 + it * TT;
    const int n = min(TT, t1 - s);
    if (tid < TT) {
      den[tid] = tid < n ? tok[(long long)(s + tid) * 2 + 0] : 1.f;
      bsc[tid] = tid < n ? tok[(long long)(s + tid) * 2 + 1] : 0.f;
      wt[tid] = dec(tid);
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
          for (int c = 0; c < DK; ++c) w = fmaf(fq[t * LDK + c], fk[j * LDK + c], w);
          for (int mm = 0; mm < DV; ++mm) dw = fmaf(aa[t * LDV + mm], vv[j * LDV + mm], dw);
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
        float a = r[c];
        for (int mm = 0; mm < DV; ++mm) a = fmaf(R[c * DV + mm], vv[j * LDV + mm], a);
        a *= dec(n - j);    // the suffix after the tile, seen from key j
        if (causal)
          for (int t = j; t < TT; ++t) a = fmaf(dW[t * (TT + 1) + j], fq[t * LDK + c], a);
        sdk[j * LDK + c] = a * phi_prime_from_phi(fk[j * LDK + c]);
      }
      for (int e = 0; e < EM; ++e) {
        const int mm = tid / TT + e * CG;
        float a = 0.f;
        for (int c = 0; c < DK; ++c) a = fmaf(R[c * DV + mm], fk[j * LDK + c], a);
        a *= dec(n - j);
        if (causal)
          for (int t = j; t < TT; ++t) a = fmaf(W[t * (TT + 1) + j], aa[t * LDV + mm], a);
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
        for (int t = 0; t < n; ++t) a = fmaf(fq[t * LDK + c] * wt[t], aa[t * LDV + m], a);
        R[c * DV + m] = a;
      }
      if (tid < DK) {
        float a = r[tid] * dec(n);
        for (int t = 0; t < n; ++t) a = fmaf(bsc[t] * wt[t], fq[t * LDK + tid], a);
        r[tid] = a;
      }
    }
    __syncthreads();
  }
}

#endif  // !LA_TILED128_ONLY

#ifdef LA_TILED128_ONLY
// ---------------------------------------------------------------------------
// dk = dv = 128 without decay: the same two sweeps with register tiles.
// Every product against the 128 x 128 state (or suffix sums) runs as 4 x 4
// outputs per thread with 16-byte shared loads of the state rows; the
// thread's rows of the state are lane, lane + 32, ... so that a warp's
// 16-byte loads of one column block hit distinct banks (rows are 132 floats
// apart). The reverse sums (sweep 1) and the state / suffix updates are 8 x 8
// tiles per thread. Same inputs, outputs and order of summation by tile as
// the kernels above.
// ---------------------------------------------------------------------------
namespace t128 {
constexpr int D = 128, LD = 132, LW = TT + 1;
constexpr size_t smem_floats() { return (size_t)D * LD + D + 4 * TT * LD + 2 * TT * LW + 2 * TT; }

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float dot4f(float4 a, float4 b, float c) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, c))));
}
// x . y over 128 floats (16-byte aligned rows)
__device__ __forceinline__ float dot128(const float* x, const float* y) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
  for (int c = 0; c < D; c += 8) {
    a0 = dot4f(ld4(x + c), ld4(y + c), a0);
    a1 = dot4f(ld4(x + c + 4), ld4(y + c + 4), a1);
  }
  return a0 + a1;
}

// The 2 x 2 block x_t . y_j, t = 2 tr + {0, 1}, j = 2 jr + {0, 1}, of rows of
// 128 floats (four 16-byte loads per 16 FMAs)
__device__ __forceinline__ void pair_dots(const float* x, const float* y, int tr, int jr, float (&o)[2][2]) {
  o[0][0] = o[0][1] = o[1][0] = o[1][1] = 0.f;
  const float* x0 = x + (2 * tr) * LD;
  const float* y0 = y + (2 * jr) * LD;
#pragma unroll 8
  for (int c = 0; c < D; c += 4) {
    const float4 a0 = ld4(x0 + c), a1 = ld4(x0 + LD + c);
    const float4 b0 = ld4(y0 + c), b1 = ld4(y0 + LD + c);
    o[0][0] = dot4f(a0, b0, o[0][0]);
    o[0][1] = dot4f(a0, b1, o[0][1]);
    o[1][0] = dot4f(a1, b0, o[1][0]);
    o[1][1] = dot4f(a1, b1, o[1][1]);
  }
}

// A tile's q, k, v and dout rows as 16-byte pieces in registers: piece
// idx = tid + i NT is row idx / (D / VPT), elements VPT (idx % (D / VPT)) ..
template <typename T>
struct TileRegs {
  static constexpr int VPT = 16 / (int)sizeof(T);      // elements per 16 bytes
  static constexpr int PER = TT * D / VPT / NT;         // pieces per thread and tensor
  uint4 r[4][PER];
};
template <typename T>
__device__ __forceinline__ void load_tile(TileRegs<T>& R, const T* q, const T* k, const T* v, const T* g, int n,
                                          int tid) {
  using TR = TileRegs<T>;
  const T* src[4] = {q, k, v, g};
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int i = 0; i < TR::PER; ++i) {
      const int idx = tid + i * NT, t = idx / (D / TR::VPT), cv = idx % (D / TR::VPT);
      R.r[x][i] = t < n ? *reinterpret_cast<const uint4*>(src[x] + (long long)t * D + cv * TR::VPT)
                        : make_uint4(0u, 0u, 0u, 0u);
    }
}
// rows [TT][LD]: phi of q and k, v and dout as they are; zero rows past n
template <typename T>
__device__ __forceinline__ void store_tile(const TileRegs<T>& R, float* fq, float* fk, float* vv, float* gg, int n,
                                           int tid) {
  using TR = TileRegs<T>;
  float* dst[4] = {fq, fk, vv, gg};
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int i = 0; i < TR::PER; ++i) {
      const int idx = tid + i * NT, t = idx / (D / TR::VPT), cv = idx % (D / TR::VPT);
      float f[TR::VPT];
      if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(R.r[x][i].x); f[1] = __uint_as_float(R.r[x][i].y);
        f[2] = __uint_as_float(R.r[x][i].z); f[3] = __uint_as_float(R.r[x][i].w);
      } else {
        const uint32_t w[4] = {R.r[x][i].x, R.r[x][i].y, R.r[x][i].z, R.r[x][i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f[2 * j] = __uint_as_float(w[j] << 16);
          f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      }
#pragma unroll
      for (int j = 0; j < TR::VPT; ++j) f[j] = t < n ? (x < 2 ? phi(f[j]) : f[j]) : 0.f;
#pragma unroll
      for (int j = 0; j < TR::VPT; j += 4)
        *reinterpret_cast<float4*>(dst[x] + t * LD + cv * TR::VPT + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
    }
}
}  // namespace t128

template <typename T>
__global__ void __launch_bounds__(NT, 1)
simt_bwd128_sweep1(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ g, T* __restrict__ dq, int N, int P, int seg_len, int causal, float eps,
                   const float* __restrict__ ws_state, long long state_words, int state_transposed,
                   float* __restrict__ ws_rev, float* __restrict__ ws_tok) {
  using namespace t128;
  extern __shared__ __align__(16) float sm[];
  float* S = sm;                  // [D][LD] state before the tile (row = key)
  float* z = S + D * LD;          // [D]
  float* fq = z + D;              // [TT][LD]
  float* fk = fq + TT * LD;
  float* vv = fk + TT * LD;
  float* aa = vv + TT * LD;       // g, then a = g / den
  float* W = aa + TT * LD;        // [TT][LW]
  float* dW = W + TT * LW;
  float* den = dW + TT * LW;      // [TT]
  float* bsc = den + TT;          // [TT]

  const long long bh = blockIdx.x;
  const int p = blockIdx.y;
  const int t0 = p * seg_len, t1 = min(N, t0 + seg_len);
  const int tid = threadIdx.x, lane = tid & 31, tg = tid >> 5;
  const int ir = tid >> 4, mr = tid & 15;           // 8 x 8 tiles: rows ir + 16 e, columns 4 mr + {0..3, 64..67}
  const T* qb = q + bh * (long long)N * D;
  const T* kb = k + bh * (long long)N * D;
  const T* vb = v + bh * (long long)N * D;
  const T* gb = g + bh * (long long)N * D;
  T* dqb = dq + bh * (long long)N * D;
  float* tok = ws_tok + bh * (long long)N * 2;
  // the state before the segment: [S | z] records, or [S^T | z | .] from the
  // tensor-core state pass
  const float* st = ws_state + (bh * P + p) * state_words;
  if (state_transposed)
    for (int i = tid; i < D * D; i += NT) S[(i % D) * LD + i / D] = st[i];
  else
    for (int i = tid; i < D * D; i += NT) S[(i / D) * LD + i % D] = st[i];
  if (tid < D) z[tid] = st[D * D + tid];
  float racc[8][8];
#pragma unroll
  for (int e = 0; e < 8; ++e)
#pragma unroll
    for (int f = 0; f < 8; ++f) racc[e][f] = 0.f;
  float rz = 0.f;
  // bf16: the next tile's inputs are loaded while a tile computes
  constexpr bool kPrefetch = sizeof(T) == 2;
  TileRegs<T> nxt;
  if (kPrefetch && t0 < t1) {
    const long long o = (long long)t0 * D;
    load_tile<T>(nxt, qb + o, kb + o, vb + o, gb + o, min(TT, t1 - t0), tid);
  }
  __syncthreads();

  for (int s = t0; s < t1; s += TT) {
    const int n = min(TT, t1 - s);
    if (!kPrefetch) {
      const long long o = (long long)s * D;
      load_tile<T>(nxt, qb + o, kb + o, vb + o, gb + o, n, tid);
    }
    store_tile<T>(nxt, fq, fk, vv, aa, n, tid);
    if (kPrefetch && s + TT < t1) {
      const long long o = (long long)(s + TT) * D;
      load_tile<T>(nxt, qb + o, kb + o, vb + o, gb + o, min(TT, t1 - s - TT), tid);
    }
    __syncthreads();
    if (causal) {
      // W_tj = phi(q_t) . phi(k_j), j <= t: 2 x 2 blocks, t = 2 (tid / 16) + .., j = 2 (tid % 16) + ..
      float o[2][2];
      pair_dots(fq, fk, tid >> 4, tid & 15, o);
#pragma unroll
      for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
          const int t = 2 * (tid >> 4) + a2, j = 2 * (tid & 15) + b2;
          W[t * LW + j] = (j <= t && t < n) ? o[a2][b2] : 0.f;
        }
      __syncthreads();
    }
    // den_t = phi(q_t) . z_prev + sum_{j <= t} W_tj + eps
    if (tid < TT) {
      const int t = tid;
      float d = dot128(fq + t * LD, z);
      if (causal)
        for (int j = 0; j <= t; ++j) d += W[t * LW + j];
      den[t] = t < n ? d + eps : 1.f;   // padding rows stay finite when eps = 0
    }
    // num[t][m] = sum_i phi(q_t)_i S[i][m] + sum_{j <= t} W_tj v_j[m]: rows 4 tg + e, columns 4 lane + f
    float num[4][4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int f = 0; f < 4; ++f) num[e][f] = 0.f;
    {
      const float* q0 = fq + (4 * tg) * LD;
#pragma unroll 4
      for (int i = 0; i < D; ++i) {
        const float4 s4 = ld4(S + i * LD + 4 * lane);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = q0[e * LD + i];
          num[e][0] = fmaf(x, s4.x, num[e][0]);
          num[e][1] = fmaf(x, s4.y, num[e][1]);
          num[e][2] = fmaf(x, s4.z, num[e][2]);
          num[e][3] = fmaf(x, s4.w, num[e][3]);
        }
      }
      if (causal) {
        for (int j = 0; j <= 4 * tg + 3; ++j) {
          const float4 v4 = ld4(vv + j * LD + 4 * lane);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float w = j <= 4 * tg + e ? W[(4 * tg + e) * LW + j] : 0.f;
            num[e][0] = fmaf(w, v4.x, num[e][0]);
            num[e][1] = fmaf(w, v4.y, num[e][1]);
            num[e][2] = fmaf(w, v4.z, num[e][2]);
            num[e][3] = fmaf(w, v4.w, num[e][3]);
          }
        }
      }
    }
    __syncthreads();   // den
    // a = g / den in place; b_t = -(a_t . num_t) / den_t (a warp holds rows 4 tg .. 4 tg + 3)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = 4 * tg + e;
      const float inv = 1.f / den[t];
      float4 g4 = ld4(aa + t * LD + 4 * lane);
      g4.x *= inv; g4.y *= inv; g4.z *= inv; g4.w *= inv;
      *reinterpret_cast<float4*>(aa + t * LD + 4 * lane) = g4;
      float part = g4.x * num[e][0] + g4.y * num[e][1] + g4.z * num[e][2] + g4.w * num[e][3];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0) {
        const float b = -part * inv;
        bsc[t] = t < n ? b : 0.f;
        if (t < n) {
          tok[(long long)(s + t) * 2 + 0] = den[t];
          tok[(long long)(s + t) * 2 + 1] = b;
        }
      }
    }
    __syncthreads();
    if (causal) {
      // dW_tj = a_t . v_j + b_t, j <= t
      float o[2][2];
      pair_dots(aa, vv, tid >> 4, tid & 15, o);
#pragma unroll
      for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
          const int t = 2 * (tid >> 4) + a2, j = 2 * (tid & 15) + b2;
          dW[t * LW + j] = (j <= t && t < n) ? o[a2][b2] + bsc[t] : 0.f;
        }
      __syncthreads();
    }
    // dphi(q_t)[i] = b_t z_i + sum_m a_t[m] S[i][m] + sum_{j <= t} dW_tj phi(k_j)_i:
    // rows 4 tg + e, columns lane + 32 f
    {
      float acc[4][4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int f = 0; f < 4; ++f) acc[e][f] = bsc[4 * tg + e] * z[lane + 32 * f];
#pragma unroll 2
      for (int m = 0; m < D; m += 4) {
        float4 a4[4], s4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) a4[e] = ld4(aa + (4 * tg + e) * LD + m);
#pragma unroll
        for (int f = 0; f < 4; ++f) s4[f] = ld4(S + (lane + 32 * f) * LD + m);
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int f = 0; f < 4; ++f) acc[e][f] = dot4f(a4[e], s4[f], acc[e][f]);
      }
      if (causal) {
        for (int j = 0; j <= 4 * tg + 3; ++j) {
          float kf[4];
#pragma unroll
          for (int f = 0; f < 4; ++f) kf[f] = fk[j * LD + lane + 32 * f];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float w = j <= 4 * tg + e ? dW[(4 * tg + e) * LW + j] : 0.f;
#pragma unroll
            for (int f = 0; f < 4; ++f) acc[e][f] = fmaf(w, kf[f], acc[e][f]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = 4 * tg + e;
        if (t < n)
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const int i = lane + 32 * f;
            dqb[(long long)(s + t) * D + i] = from_f32<T>(acc[e][f] * phi_prime_from_phi(fq[t * LD + i]));
          }
      }
    }
    // reverse sums over the segment: R += phi(Q)^T a, r += sum_t b_t phi(q_t)
    for (int t = 0; t < n; ++t) {
      const float4 a0 = ld4(aa + t * LD + 4 * mr), a1 = ld4(aa + t * LD + 64 + 4 * mr);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = fq[t * LD + ir + 16 * e];
        racc[e][0] = fmaf(x, a0.x, racc[e][0]); racc[e][1] = fmaf(x, a0.y, racc[e][1]);
        racc[e][2] = fmaf(x, a0.z, racc[e][2]); racc[e][3] = fmaf(x, a0.w, racc[e][3]);
        racc[e][4] = fmaf(x, a1.x, racc[e][4]); racc[e][5] = fmaf(x, a1.y, racc[e][5]);
        racc[e][6] = fmaf(x, a1.z, racc[e][6]); racc[e][7] = fmaf(x, a1.w, racc[e][7]);
      }
    }
    if (tid < D)
      for (int t = 0; t < n; ++t) rz = fmaf(bsc[t], fq[t * LD + tid], rz);
    if (causal) {
      __syncthreads();   // every read of S and z for this tile is done
      // S += phi(K)^T V, z += sum phi(k)
      float sacc[8][8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float4 s0 = ld4(S + (ir + 16 * e) * LD + 4 * mr), s1 = ld4(S + (ir + 16 * e) * LD + 64 + 4 * mr);
        sacc[e][0] = s0.x; sacc[e][1] = s0.y; sacc[e][2] = s0.z; sacc[e][3] = s0.w;
        sacc[e][4] = s1.x; sacc[e][5] = s1.y; sacc[e][6] = s1.z; sacc[e][7] = s1.w;
      }
      for (int t = 0; t < n; ++t) {
        const float4 v0 = ld4(vv + t * LD + 4 * mr), v1 = ld4(vv + t * LD + 64 + 4 * mr);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = fk[t * LD + ir + 16 * e];
          sacc[e][0] = fmaf(x, v0.x, sacc[e][0]); sacc[e][1] = fmaf(x, v0.y, sacc[e][1]);
          sacc[e][2] = fmaf(x, v0.z, sacc[e][2]); sacc[e][3] = fmaf(x, v0.w, sacc[e][3]);
          sacc[e][4] = fmaf(x, v1.x, sacc[e][4]); sacc[e][5] = fmaf(x, v1.y, sacc[e][5]);
          sacc[e][6] = fmaf(x, v1.z, sacc[e][6]); sacc[e][7] = fmaf(x, v1.w, sacc[e][7]);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        *reinterpret_cast<float4*>(S + (ir + 16 * e) * LD + 4 * mr) =
            make_float4(sacc[e][0], sacc[e][1], sacc[e][2], sacc[e][3]);
        *reinterpret_cast<float4*>(S + (ir + 16 * e) * LD + 64 + 4 * mr) =
            make_float4(sacc[e][4], sacc[e][5], sacc[e][6], sacc[e][7]);
      }
      if (tid < D) {
        float a = z[tid];
        for (int t = 0; t < n; ++t) a += fk[t * LD + tid];
        z[tid] = a;
      }
    }
    __syncthreads();
  }
  float* o = ws_rev + (bh * P + p) * (long long)(D * D + D);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    *reinterpret_cast<float4*>(o + (ir + 16 * e) * D + 4 * mr) = make_float4(racc[e][0], racc[e][1], racc[e][2], racc[e][3]);
    *reinterpret_cast<float4*>(o + (ir + 16 * e) * D + 64 + 4 * mr) =
        make_float4(racc[e][4], racc[e][5], racc[e][6], racc[e][7]);
  }
  if (tid < D) o[D * D + tid] = rz;
}

template <typename T>
__global__ void __launch_bounds__(NT, 1)
simt_bwd128_sweep2(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ g, T* __restrict__ dk_, T* __restrict__ dv_, int N, int P, int seg_len,
                   int causal, const float* __restrict__ ws_rev, const float* __restrict__ ws_tok) {
  using namespace t128;
  extern __shared__ __align__(16) float sm[];
  float* R = sm;                  // [D][LD] suffix sums after the tile (row = key)
  float* r = R + D * LD;          // [D]
  float* fq = r + D;
  float* fk = fq + TT * LD;
  float* vv = fk + TT * LD;
  float* aa = vv + TT * LD;       // a = g / den
  float* W = aa + TT * LD;
  float* dW = W + TT * LW;
  float* den = dW + TT * LW;
  float* bsc = den + TT;

  const long long bh = blockIdx.x;
  const int p = blockIdx.y;
  const int t0 = p * seg_len, t1 = min(N, t0 + seg_len);
  const int tid = threadIdx.x, lane = tid & 31, tg = tid >> 5;
  const int ir = tid >> 4, mr = tid & 15;
  const T* qb = q + bh * (long long)N * D;
  const T* kb = k + bh * (long long)N * D;
  const T* vb = v + bh * (long long)N * D;
  const T* gb = g + bh * (long long)N * D;
  T* dkb = dk_ + bh * (long long)N * D;
  T* dvb = dv_ + bh * (long long)N * D;
  const float* tok = ws_tok + bh * (long long)N * 2;
  const float* st = ws_rev + (bh * P + p) * (long long)(D * D + D);
  for (int i = tid; i < D * D; i += NT) R[(i / D) * LD + i % D] = st[i];
  if (tid < D) r[tid] = st[D * D + tid];
  __syncthreads();

  const int ntiles = (t1 - t0 + TT - 1) / TT;
  constexpr bool kPrefetch = sizeof(T) == 2;
  TileRegs<T> nxt;
  if (kPrefetch && ntiles > 0) {
    const int s = t0 + (ntiles - 1) * TT;
    const long long o = (long long)s * D;
    load_tile<T>(nxt, qb + o, kb + o, vb + o, gb + o, min(TT, t1 - s), tid);
  }
  for (int it = ntiles - 1; it >= 0; --it) {
    const int s = t0 + it * TT;
    const int n = min(TT, t1 - s);
    if (tid < TT) {
      den[tid] = tid < n ? tok[(long long)(s + tid) * 2 + 0] : 1.f;
      bsc[tid] = tid < n ? tok[(long long)(s + tid) * 2 + 1] : 0.f;
    }
    if (!kPrefetch) {
      const long long o = (long long)s * D;
      load_tile<T>(nxt, qb + o, kb + o, vb + o, gb + o, n, tid);
    }
    store_tile<T>(nxt, fq, fk, vv, aa, n, tid);
    if (kPrefetch && it > 0) {
      // the tile before this one (the sweep runs backwards): always whole
      const long long o = (long long)(s - TT) * D;
      load_tile<T>(nxt, qb + o, kb + o, vb + o, gb + o, TT, tid);
    }
    __syncthreads();   // den visible
    for (int idx = tid; idx < TT * D; idx += NT) {
      const int t = idx / D, c = idx % D;
      aa[t * LD + c] /= den[t];
    }
    __syncthreads();
    if (causal) {
      float o[2][2], od[2][2];
      pair_dots(fq, fk, tid >> 4, tid & 15, o);
      pair_dots(aa, vv, tid >> 4, tid & 15, od);
#pragma unroll
      for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
          const int t = 2 * (tid >> 4) + a2, j = 2 * (tid & 15) + b2;
          const bool keep = j <= t && t < n;
          W[t * LW + j] = keep ? o[a2][b2] : 0.f;
          dW[t * LW + j] = keep ? od[a2][b2] + bsc[t] : 0.f;
        }
      __syncthreads();
    }
    // dphi(k_j)[i] = r_i + sum_m R[i][m] v_j[m] + sum_{t >= j} dW_tj phi(q_t)_i:
    // rows j = 4 tg + e, columns i = lane + 32 f
    {
      float acc[4][4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int f = 0; f < 4; ++f) acc[e][f] = r[lane + 32 * f];
#pragma unroll 2
      for (int m = 0; m < D; m += 4) {
        float4 v4[4], r4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v4[e] = ld4(vv + (4 * tg + e) * LD + m);
#pragma unroll
        for (int f = 0; f < 4; ++f) r4[f] = ld4(R + (lane + 32 * f) * LD + m);
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int f = 0; f < 4; ++f) acc[e][f] = dot4f(v4[e], r4[f], acc[e][f]);
      }
      if (causal) {
        for (int t = 4 * tg; t < TT; ++t) {
          float qf[4];
#pragma unroll
          for (int f = 0; f < 4; ++f) qf[f] = fq[t * LD + lane + 32 * f];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * tg + e;
            const float w = t >= j ? dW[t * LW + j] : 0.f;
#pragma unroll
            for (int f = 0; f < 4; ++f) acc[e][f] = fmaf(w, qf[f], acc[e][f]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * tg + e;
        if (j < n)
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const int i = lane + 32 * f;
            dkb[(long long)(s + j) * D + i] = from_f32<T>(acc[e][f] * phi_prime_from_phi(fk[j * LD + i]));
          }
      }
    }
    // dv_j[m] = sum_i R[i][m] phi(k_j)_i + sum_{t >= j} W_tj a_t[m]: rows j = 4 tg + e, columns 4 lane + f
    {
      float acc[4][4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int f = 0; f < 4; ++f) acc[e][f] = 0.f;
      const float* k0 = fk + (4 * tg) * LD;
#pragma unroll 4
      for (int i = 0; i < D; ++i) {
        const float4 r4 = ld4(R + i * LD + 4 * lane);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = k0[e * LD + i];
          acc[e][0] = fmaf(x, r4.x, acc[e][0]);
          acc[e][1] = fmaf(x, r4.y, acc[e][1]);
          acc[e][2] = fmaf(x, r4.z, acc[e][2]);
          acc[e][3] = fmaf(x, r4.w, acc[e][3]);
        }
      }
      if (causal) {
        for (int t = 4 * tg; t < TT; ++t) {
          const float4 a4 = ld4(aa + t * LD + 4 * lane);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * tg + e;
            const float w = t >= j ? W[t * LW + j] : 0.f;
            acc[e][0] = fmaf(w, a4.x, acc[e][0]);
            acc[e][1] = fmaf(w, a4.y, acc[e][1]);
            acc[e][2] = fmaf(w, a4.z, acc[e][2]);
            acc[e][3] = fmaf(w, a4.w, acc[e][3]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * tg + e;
        if (j < n)
#pragma unroll
          for (int f = 0; f < 4; ++f) dvb[(long long)(s + j) * D + 4 * lane + f] = from_f32<T>(acc[e][f]);
      }
    }
    if (causal) {
      __syncthreads();   // every read of R and r for this tile is done
      // R += phi(Q)^T a, r += sum_t b_t phi(q_t): the suffix at the tile's first token
      float racc[8][8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float4 s0 = ld4(R + (ir + 16 * e) * LD + 4 * mr), s1 = ld4(R + (ir + 16 * e) * LD + 64 + 4 * mr);
        racc[e][0] = s0.x; racc[e][1] = s0.y; racc[e][2] = s0.z; racc[e][3] = s0.w;
        racc[e][4] = s1.x; racc[e][5] = s1.y; racc[e][6] = s1.z; racc[e][7] = s1.w;
      }
      for (int t = 0; t < n; ++t) {
        const float4 a0 = ld4(aa + t * LD + 4 * mr), a1 = ld4(aa + t * LD + 64 + 4 * mr);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = fq[t * LD + ir + 16 * e];
          racc[e][0] = fmaf(x, a0.x, racc[e][0]); racc[e][1] = fmaf(x, a0.y, racc[e][1]);
          racc[e][2] = fmaf(x, a0.z, racc[e][2]); racc[e][3] = fmaf(x, a0.w, racc[e][3]);
          racc[e][4] = fmaf(x, a1.x, racc[e][4]); racc[e][5] = fmaf(x, a1.y, racc[e][5]);
          racc[e][6] = fmaf(x, a1.z, racc[e][6]); racc[e][7] = fmaf(x, a1.w, racc[e][7]);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        *reinterpret_cast<float4*>(R + (ir + 16 * e) * LD + 4 * mr) =
            make_float4(racc[e][0], racc[e][1], racc[e][2], racc[e][3]);
        *reinterpret_cast<float4*>(R + (ir + 16 * e) * LD + 64 + 4 * mr) =
            make_float4(racc[e][4], racc[e][5], racc[e][6], racc[e][7]);
      }
      if (tid < D) {
        float a = r[tid];
        for (int t = 0; t < n; ++t) a = fmaf(bsc[t], fq[t * LD + tid], a);
        r[tid] = a;
      }
    }
    __syncthreads();
  }
}

// dk = dv = 128 without decay: the state pass (on the tensor cores for bf16
// inputs: the forward's state kernel, records [S^T | z | .]), the scans and
// the register-tiled sweeps
template <typename T>
cudaError_t launch_bwd128(const BwdArgs& a, const FwdArgs& f) {
  constexpr int D = 128;
  const long long words = state_words(D, D);
  const bool tc_state = std::is_same<T, __nv_bfloat16>::value && a.plan.F == 1 && device_status_ptr() != nullptr;
  const long long swords = tc_state ? (long long)D * D + 2 * D : words;
  prof_begin(LA_SPAN_BWD_STATE, a.stream);
  cudaError_t err = tc_state ? tc_segment_state(f) : simt_segment_state(f);
  if (err == cudaSuccess)
    err = segment_scan(a.ws_state, a.BH, a.plan.P, swords, a.causal ? SCAN_EXCLUSIVE_FWD : SCAN_TOTAL, nullptr,
                       nullptr, D, D, a.stream, nullptr, 1, a.plan.seg_len, a.N);
  prof_end(LA_SPAN_BWD_STATE, a.stream);
  if (err != cudaSuccess) return err;
  dim3 grid(a.BH, a.plan.P);
  constexpr size_t smem = sizeof(float) * t128::smem_floats();
  auto s1 = simt_bwd128_sweep1<T>;
  auto s2 = simt_bwd128_sweep2<T>;
  err = cudaFuncSetAttribute(s1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err == cudaSuccess) err = cudaFuncSetAttribute(s2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  prof_begin(LA_SPAN_BWD_SWEEP1, a.stream);
  s1<<<grid, NT, smem, a.stream>>>((const T*)a.q, (const T*)a.k, (const T*)a.v, (const T*)a.dout, (T*)a.dq, a.N,
                                   a.plan.P, a.plan.seg_len, a.causal, a.eps, a.ws_state, swords, tc_state ? 1 : 0,
                                   a.ws_rev, a.ws_tok);
  prof_end(LA_SPAN_BWD_SWEEP1, a.stream);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  note_launch();
  prof_begin(LA_SPAN_BWD_SCAN, a.stream);
  err = segment_scan(a.ws_rev, a.BH, a.plan.P, words, a.causal ? SCAN_EXCLUSIVE_REV : SCAN_TOTAL, nullptr, nullptr,
                     D, D, a.stream, nullptr, 1, a.plan.seg_len, a.N);
  prof_end(LA_SPAN_BWD_SCAN, a.stream);
  if (err != cudaSuccess) return err;
  prof_begin(LA_SPAN_BWD_SWEEP2, a.stream);
  s2<<<grid, NT, smem, a.stream>>>((const T*)a.q, (const T*)a.k, (const T*)a.v, (const T*)a.dout, (T*)a.dk_,
                                   (T*)a.dv_, a.N, a.plan.P, a.plan.seg_len, a.causal, a.ws_rev, a.ws_tok);
  prof_end(LA_SPAN_BWD_SWEEP2, a.stream);
  err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

#endif  // LA_TILED128_ONLY

#ifndef LA_TILED128_ONLY
template <int DK, int DV, typename T>
cudaError_t launch_bwd(const BwdArgs& a) {
  FwdArgs f{};
  f.q = a.q; f.k = a.k; f.v = a.v; f.out = nullptr;
  f.BH = a.BH; f.N = a.N; f.dk = a.dk; f.dv = a.dv; f.causal = a.causal;
  f.eps = a.eps; f.dtype = a.dtype; f.ws_state = a.ws_state; f.plan = a.plan;
  f.stream = a.stream;
  f.alpha = a.alpha; f.H = a.H;
  if constexpr (DK == 128 && DV == 128) {
    if (a.alpha == nullptr) return simt_backward_tiled128(a);
  }
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

#endif  // !LA_TILED128_ONLY

}  // namespace

#ifdef LA_TILED128_ONLY
cudaError_t simt_backward_tiled128(const BwdArgs& a) {
  FwdArgs f{};
  f.q = a.q; f.k = a.k; f.v = a.v; f.out = nullptr;
  f.BH = a.BH; f.N = a.N; f.dk = a.dk; f.dv = a.dv; f.causal = a.causal;
  f.eps = a.eps; f.dtype = a.dtype; f.ws_state = a.ws_state; f.plan = a.plan;
  f.stream = a.stream;
  return a.dtype == LA_BF16 ? launch_bwd128<__nv_bfloat16>(a, f) : launch_bwd128<float>(a, f);
}
#else
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

#endif  // LA_TILED128_ONLY

}  // namespace la
