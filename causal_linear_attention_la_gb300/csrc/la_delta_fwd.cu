// Delta rule over whole sequences, chunk by chunk (CUDA cores, fp32).
//
// The update of "Linear Attention, 곱의 순서를 바꾸면 생기는 일" (paragraph on
// 델타 규칙), token by token: read the state with the key, write only the
// difference to the value, read with the query,
//   u_t = S_{t-1}^T k_t,  S_t = S_{t-1} + k_t (v_t - u_t)^T,  o_t = S_t^T q_t.
// Writing u'_t = v_t - S_{t-1}^T k_t for the increment of token t, a chunk of
// C tokens starting from S_0 satisfies S_t = S_0 + sum_{j <= t} k_j u'_j^T, so
//   u'_t = v_t - S_0^T k_t - sum_{j < t} (k_j . k_t) u'_j,
// i.e. (I + A) U' = V - K S_0 with A = (K K^T) strictly below the diagonal: a
// unit lower-triangular system (the WY form of the chunk's product of
// rank-one updates). Then
//   O = Q S_0 + (Q K^T masked to j <= t) U',   S_C = S_0 + K^T U'.
//
// Every column of S evolves on its own (column m of S_t depends only on
// column m of the values), so a head's state is split into blocks of DB
// columns, one CTA each; the CTAs of a head share nothing but their keys and
// queries. Per 32-token chunk a CTA runs
//   1. one register-tiled pass [K ; Q] x [S_0 block | K^T] (64 x (DB + 32),
//      depth d): R = V - K S_0, P = Q S_0, A = K K^T and Q K^T together;
//   2. the triangular solve (I + A) U' = R, one lane per token: at step j
//      lane j holds its final u'_j and the later lanes subtract a_tj u'_j
//      (a warp shuffle), DB / 8 columns per warp;
//   3. O = P + (Q K^T masked) U' (the threads that hold P) and
//      S_0 += K^T U' (the state block lives in registers, 4 x 4 per thread).
// The next chunk's inputs are loaded into registers while a chunk computes.
#include "la_internal.cuh"
#include "la_variants.cuh"

namespace la {

namespace {

constexpr int NT = 256;   // threads
constexpr int CT = 32;    // tokens per chunk: one per lane in the solve

template <int D>
struct DeltaTile {
  static constexpr int DB = D < 32 ? D : 32;    // state columns per CTA
  static constexpr int NB = D / DB;             // CTAs per head
  static constexpr int CGN = (DB + CT) / 4;     // column groups of pass 1
  static constexpr int LDA = 2 * CT;            // row c of [K^T | Q^T]
  static constexpr int LDR = D + 4;             // token-major K row
  static constexpr int LDV = DB + 1;            // value block row
  static constexpr int LDU = DB + 4;            // R, then U'
  static constexpr int LDP = CT + 1;            // K K^T and Q K^T rows
  static constexpr int KQT = 0;                          // [D][LDA]
  static constexpr int KR = KQT + D * LDA;               // [CT][LDR]
  static constexpr int SB = KR + CT * LDR;               // [D][DB] state block
  static constexpr int VS = SB + D * DB;                 // [CT][LDV]
  static constexpr int US = VS + CT * LDV;               // [CT][LDU]
  static constexpr int AS = US + CT * LDU;               // [CT][LDP]
  static constexpr int QKS = AS + CT * LDP;              // [CT][LDP]
  static constexpr int FLOATS = QKS + CT * LDP;
  static_assert(KR % 4 == 0 && SB % 4 == 0 && US % 4 == 0 && LDR % 4 == 0 && LDU % 4 == 0,
                "float4 rows");
};

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& r, float* f) {
  if constexpr (sizeof(T) == 4) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
  } else {
    const unsigned w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float a, float b, float c, float d) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 w;
    w.x = *reinterpret_cast<unsigned*>(&lo);
    w.y = *reinterpret_cast<unsigned*>(&hi);
    *reinterpret_cast<uint2*>(p) = w;
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(NT, 2)
delta_chunk_kernel(float* __restrict__ S, const T* __restrict__ q, const T* __restrict__ k,
                   const T* __restrict__ v, T* __restrict__ out, int N) {
  using L = DeltaTile<D>;
  constexpr int DB = L::DB, NB = L::NB, CGN = L::CGN;
  constexpr int LDA = L::LDA, LDR = L::LDR, LDV = L::LDV, LDU = L::LDU, LDP = L::LDP;
  constexpr int VEC = 16 / (int)sizeof(T);         // inputs per 16-byte load
  constexpr int KITEMS = CT * (D / VEC);           // 16-byte pieces of a q or k chunk
  constexpr int KPER = (KITEMS + NT - 1) / NT;
  constexpr int VITEMS = CT * (DB / VEC);          // of the chunk's value block
  constexpr int VPER = (VITEMS + NT - 1) / NT;
  constexpr int CPW = DB / 8;                      // solve: columns per warp
  constexpr int UPD = D * DB / 16;                 // threads holding a 4 x 4 state tile
  extern __shared__ __align__(16) float sm[];
  float* KQt = sm + L::KQT;
  float* Kr = sm + L::KR;
  float* Sb = sm + L::SB;
  float* Vs = sm + L::VS;
  float* Us = sm + L::US;
  float* As = sm + L::AS;
  float* QKs = sm + L::QKS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long bh = blockIdx.x / NB;
  const int col0 = (blockIdx.x % NB) * DB;
  float* Sg = S + bh * (long long)D * D + col0;
  const T* qb = q + bh * (long long)N * D;
  const T* kb = k + bh * (long long)N * D;
  const T* vb = v + bh * (long long)N * D + col0;
  T* ob = out + bh * (long long)N * D + col0;

  // state tile of this thread: rows c0..c0+3, columns m0..m0+3 of the block
  const int s_c0 = 4 * (tid / (DB / 4)), s_m0 = 4 * (tid % (DB / 4));
  float st[4][4];
  if (tid < UPD) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 r = *reinterpret_cast<const float4*>(Sg + (long long)(s_c0 + i) * D + s_m0);
      st[i][0] = r.x; st[i][1] = r.y; st[i][2] = r.z; st[i][3] = r.w;
      *reinterpret_cast<float4*>(Sb + (s_c0 + i) * DB + s_m0) = r;
    }
  }

  // pass-1 tile: rows r0..r0+3 of [K ; Q], columns g0..g0+3 of [S_0 block | K^T]
  const int p_rg = tid / CGN, p_cg = tid % CGN;
  const bool p_on = tid < 16 * CGN;
  const int p_r0 = 4 * p_rg;
  const bool p_state = p_cg < DB / 4;              // column group inside the state block
  const int p_g0 = p_state ? 4 * p_cg : 4 * (p_cg - DB / 4);
  const float* pb = p_state ? Sb + p_g0 : KQt + p_g0;
  const int pstride = p_state ? DB : LDA;

  uint4 kr[KPER], qr[KPER], vr[VPER];
  auto prefetch = [&](int s) {
#pragma unroll
    for (int i = 0; i < KPER; ++i) {
      const int idx = tid + i * NT, t = idx % CT, g = idx / CT;
      const bool in = idx < KITEMS && s + t < N;
      const long long off = (long long)(s + t) * D + g * VEC;
      kr[i] = in ? __ldg(reinterpret_cast<const uint4*>(kb + off)) : make_uint4(0, 0, 0, 0);
      qr[i] = in ? __ldg(reinterpret_cast<const uint4*>(qb + off)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < VPER; ++i) {
      const int idx = tid + i * NT, t = idx % CT, g = idx / CT;
      const bool in = idx < VITEMS && s + t < N;
      vr[i] = in ? __ldg(reinterpret_cast<const uint4*>(vb + (long long)(s + t) * D + g * VEC))
                 : make_uint4(0, 0, 0, 0);
    }
  };
  prefetch(0);

  for (int s = 0; s < N; s += CT) {
    const int n = min(CT, N - s);
    __syncthreads();   // the previous chunk's readers of Kr, Us and its Sb writes are done
#pragma unroll
    for (int i = 0; i < KPER; ++i) {
      const int idx = tid + i * NT, t = idx % CT, g = idx / CT;
      if (idx < KITEMS) {
        float f[VEC], h[VEC];
        unpack16<T>(kr[i], f);
        unpack16<T>(qr[i], h);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          KQt[(g * VEC + j) * LDA + t] = f[j];
          KQt[(g * VEC + j) * LDA + CT + t] = h[j];
        }
#pragma unroll
        for (int j = 0; j < VEC; j += 4)
          *reinterpret_cast<float4*>(Kr + t * LDR + g * VEC + j) =
              make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
      }
    }
#pragma unroll
    for (int i = 0; i < VPER; ++i) {
      const int idx = tid + i * NT, t = idx % CT, g = idx / CT;
      if (idx < VITEMS) {
        float f[VEC];
        unpack16<T>(vr[i], f);
#pragma unroll
        for (int j = 0; j < VEC; ++j) Vs[t * LDV + g * VEC + j] = f[j];
      }
    }
    if (s + CT < N) prefetch(s + CT);
    __syncthreads();

    // 1. [K ; Q] x [S_0 block | K^T]
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    if (p_on) {
      const float* pa = KQt + p_r0;
#pragma unroll 8
      for (int c = 0; c < D; ++c) {
        const float4 a = *reinterpret_cast<const float4*>(pa + c * LDA);
        const float4 b = *reinterpret_cast<const float4*>(pb + c * pstride);
        const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      if (p_r0 < CT) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (p_state) Us[(p_r0 + i) * LDU + p_g0 + j] = Vs[(p_r0 + i) * LDV + p_g0 + j] - acc[i][j];
            else As[(p_r0 + i) * LDP + p_g0 + j] = acc[i][j];
          }
      } else if (!p_state) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) QKs[(p_r0 - CT + i) * LDP + p_g0 + j] = acc[i][j];
      }
    }
    __syncthreads();

    // 2. (I + A) U' = R: lane t holds row t of CPW columns
    {
      float r[CPW];
#pragma unroll
      for (int i = 0; i < CPW; ++i) r[i] = Us[lane * LDU + warp * CPW + i];
#pragma unroll
      for (int j = 0; j < CT - 1; ++j) {
        const float a = As[lane * LDP + j];
#pragma unroll
        for (int i = 0; i < CPW; ++i) {
          const float x = __shfl_sync(0xffffffffu, r[i], j);
          if (j < lane) r[i] = fmaf(-a, x, r[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < CPW; ++i) Us[lane * LDU + warp * CPW + i] = r[i];
    }
    __syncthreads();

    // 3a. O = Q S_0 + (Q K^T masked) U', by the threads holding Q S_0
    if (p_on && p_r0 >= CT && p_state) {
      const int t0 = p_r0 - CT;
      const int jend = min(t0 + 4, n);
      for (int j = 0; j < jend; ++j) {
        const float4 u = *reinterpret_cast<const float4*>(Us + j * LDU + p_g0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float w = j <= t0 + i ? QKs[(t0 + i) * LDP + j] : 0.f;
          acc[i][0] = fmaf(w, u.x, acc[i][0]);
          acc[i][1] = fmaf(w, u.y, acc[i][1]);
          acc[i][2] = fmaf(w, u.z, acc[i][2]);
          acc[i][3] = fmaf(w, u.w, acc[i][3]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (t0 + i < n)
          store4<T>(ob + (long long)(s + t0 + i) * D + p_g0, acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
    // 3b. S_0 += K^T U' on the register tile, copied to Sb for the next chunk
    if (tid < UPD) {
      for (int t = 0; t < n; ++t) {
        const float4 kk = *reinterpret_cast<const float4*>(Kr + t * LDR + s_c0);
        const float4 u = *reinterpret_cast<const float4*>(Us + t * LDU + s_m0);
        const float kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          st[i][0] = fmaf(kv[i], u.x, st[i][0]);
          st[i][1] = fmaf(kv[i], u.y, st[i][1]);
          st[i][2] = fmaf(kv[i], u.z, st[i][2]);
          st[i][3] = fmaf(kv[i], u.w, st[i][3]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(Sb + (s_c0 + i) * DB + s_m0) =
            make_float4(st[i][0], st[i][1], st[i][2], st[i][3]);
    }
  }
  if (tid < UPD) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(Sg + (long long)(s_c0 + i) * D + s_m0) =
          make_float4(st[i][0], st[i][1], st[i][2], st[i][3]);
  }
}

template <int D, typename T>
cudaError_t launch_delta_chunks(const VariantArgs& a) {
  using L = DeltaTile<D>;
  constexpr size_t smem = sizeof(float) * L::FLOATS;
  auto kern = delta_chunk_kernel<D, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)a.BH * L::NB;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)grid, NT, smem, a.stream>>>(a.S, (const T*)a.q, (const T*)a.k, (const T*)a.v,
                                                (T*)a.out, a.ntok);
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
