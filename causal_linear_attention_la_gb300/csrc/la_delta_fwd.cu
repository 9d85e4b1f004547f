// Delta rule over whole sequences, chunk by chunk (CUDA cores, fp32).
//
// The update of "Linear Attention, 곱의 순서를 바꾸면 생기는 일" (paragraph on
// 델타 규칙), token by token: read the state with the key, write only the
// difference to the value, read with the query,
//   u_t = S_{t-1}^T k_t,  S_t = S_{t-1} + k_t (v_t - u_t)^T,  o_t = S_t^T q_t.
// Writing u'_t = v_t - S_{t-1}^T k_t for the increment of token t, a chunk of C
// tokens starting from S_0 satisfies S_t = S_0 + sum_{j <= t} k_j u'_j^T, so
//   u'_t = v_t - S_0^T k_t - sum_{j < t} (k_j . k_t) u'_j,
// i.e. (I + A) U' = V - K S_0 with A = (K K^T) strictly below the diagonal:
// a unit lower-triangular system. With W = (I + A)^-1 K and U~ = (I + A)^-1 V
// (forward substitution, the WY form of the chunk's product of rank-one
// updates), U' = U~ - W S_0, and
//   O = Q S_0 + (Q K^T masked to j <= t) U',   S_C = S_0 + K^T U'.
// The chunk is then dense matrix products plus one triangular solve whose
// rows depend on each other but whose columns do not: thread c solves
// column c of [W | U~] alone, with no barrier between rows.
//
// One CTA per (batch, head) runs its chunks in order, the fp32 state in
// shared memory for the whole sequence; dk = dv in {16, 32, 64, 128}.
#include "la_internal.cuh"
#include "la_variants.cuh"

namespace la {

namespace {

constexpr int NT = 256;   // threads
constexpr int CT = 32;    // tokens per chunk

template <int D>
struct DeltaSmem {
  static constexpr int LD = D + 1;                      // padded rows
  static constexpr int S_OFF = 0;                       // [D][D] state
  static constexpr int K_OFF = S_OFF + D * D;           // [CT][LD] keys
  static constexpr int Q_OFF = K_OFF + CT * LD;         // [CT][LD] queries
  static constexpr int W_OFF = Q_OFF + CT * LD;         // [CT][LD] W = (I + A)^-1 K
  static constexpr int U_OFF = W_OFF + CT * LD;         // [CT][LD] V, then U~, then U'
  static constexpr int A_OFF = U_OFF + CT * LD;         // [CT][CT + 1] k_t . k_j, j < t
  static constexpr int QK_OFF = A_OFF + CT * (CT + 1);  // [CT][CT + 1] q_t . k_j, j <= t
  static constexpr int FLOATS = QK_OFF + CT * (CT + 1);
};

template <int D, typename T>
__global__ void __launch_bounds__(NT)
delta_chunk_kernel(float* __restrict__ S, const T* __restrict__ q, const T* __restrict__ k,
                   const T* __restrict__ v, T* __restrict__ out, int N) {
  using L = DeltaSmem<D>;
  constexpr int LD = L::LD;
  constexpr int RG = NT / D;          // row groups: thread (m, g) = (tid % D, tid / D)
  extern __shared__ float sm[];
  float* St = sm + L::S_OFF;
  float* Kc = sm + L::K_OFF;
  float* Qc = sm + L::Q_OFF;
  float* Wc = sm + L::W_OFF;
  float* Uc = sm + L::U_OFF;
  float* Am = sm + L::A_OFF;
  float* QK = sm + L::QK_OFF;

  const long long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int m = tid % D, g = tid / D;
  float* Sg = S + bh * (long long)D * D;
  const T* qb = q + bh * (long long)N * D;
  const T* kb = k + bh * (long long)N * D;
  const T* vb = v + bh * (long long)N * D;
  T* ob = out + bh * (long long)N * D;
  for (int i = tid; i < D * D; i += NT) St[i] = Sg[i];

  for (int s = 0; s < N; s += CT) {
    const int n = min(CT, N - s);
    __syncthreads();   // the previous chunk is done with every buffer
    for (int idx = tid; idx < CT * D; idx += NT) {
      const int t = idx / D, c = idx % D;
      const bool in = t < n;
      Kc[t * LD + c] = in ? to_f32<T>(kb[(long long)(s + t) * D + c]) : 0.f;
      Qc[t * LD + c] = in ? to_f32<T>(qb[(long long)(s + t) * D + c]) : 0.f;
      Uc[t * LD + c] = in ? to_f32<T>(vb[(long long)(s + t) * D + c]) : 0.f;
    }
    __syncthreads();
    // k_t . k_j (j < t) and q_t . k_j (j <= t)
    for (int idx = tid; idx < CT * CT; idx += NT) {
      const int t = idx / CT, j = idx % CT;
      float a = 0.f, b = 0.f;
      if (j <= t && t < n) {
        for (int c = 0; c < D; ++c) {
          const float kj = Kc[j * LD + c];
          a = fmaf(Kc[t * LD + c], kj, a);
          b = fmaf(Qc[t * LD + c], kj, b);
        }
      }
      Am[t * (CT + 1) + j] = j < t ? a : 0.f;
      QK[t * (CT + 1) + j] = b;
    }
    __syncthreads();
    // (I + A) [W | U~] = [K | V] by forward substitution, one column per
    // thread (columns 0..D-1 of W, D..2D-1 of U~); rows past n stay zero
    for (int col = tid; col < 2 * D; col += NT) {
      const bool isw = col < D;
      const int c = isw ? col : col - D;
      float* X = isw ? Wc : Uc;
      const float* rhs = isw ? Kc : Uc;       // U~ overwrites V row by row
      for (int t = 0; t < n; ++t) {
        float x = rhs[t * LD + c];
        for (int j = 0; j < t; ++j) x = fmaf(-Am[t * (CT + 1) + j], X[j * LD + c], x);
        X[t * LD + c] = x;
      }
      for (int t = n; t < CT; ++t) X[t * LD + c] = 0.f;
    }
    __syncthreads();
    // U' = U~ - W S_0 (in place), thread (m, g) for rows t = g, g + RG, ...
    for (int t = g; t < CT; t += RG) {
      float a = Uc[t * LD + m];
      for (int c = 0; c < D; ++c) a = fmaf(-Wc[t * LD + c], St[c * D + m], a);
      Uc[t * LD + m] = a;
    }
    __syncthreads();
    // O = Q S_0 + (Q K^T masked) U'
    for (int t = g; t < n; t += RG) {
      float a = 0.f;
      for (int c = 0; c < D; ++c) a = fmaf(Qc[t * LD + c], St[c * D + m], a);
      for (int j = 0; j <= t; ++j) a = fmaf(QK[t * (CT + 1) + j], Uc[j * LD + m], a);
      ob[(long long)(s + t) * D + m] = from_f32<T>(a);
    }
    __syncthreads();   // every read of S_0 is done
    // S <- S_0 + K^T U'
    for (int c = g; c < D; c += RG) {
      float a = St[c * D + m];
      for (int t = 0; t < n; ++t) a = fmaf(Kc[t * LD + c], Uc[t * LD + m], a);
      St[c * D + m] = a;
    }
  }
  __syncthreads();
  for (int i = tid; i < D * D; i += NT) Sg[i] = St[i];
}

template <int D, typename T>
cudaError_t launch_delta_chunks(const VariantArgs& a) {
  constexpr size_t smem = sizeof(float) * DeltaSmem<D>::FLOATS;
  auto kern = delta_chunk_kernel<D, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<a.BH, NT, smem, a.stream>>>(a.S, (const T*)a.q, (const T*)a.k, (const T*)a.v, (T*)a.out, a.ntok);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace

cudaError_t forward_delta_chunked(const VariantArgs& a) {
  if (a.dk != a.dv) return cudaErrorInvalidValue;
  const bool bf = a.dtype == LA_BF16;
  switch (a.dk) {
    case 16: return bf ? launch_delta_chunks<16, __nv_bfloat16>(a) : launch_delta_chunks<16, float>(a);
    case 32: return bf ? launch_delta_chunks<32, __nv_bfloat16>(a) : launch_delta_chunks<32, float>(a);
    case 64: return bf ? launch_delta_chunks<64, __nv_bfloat16>(a) : launch_delta_chunks<64, float>(a);
    case 128: return bf ? launch_delta_chunks<128, __nv_bfloat16>(a) : launch_delta_chunks<128, float>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace la
