// Tensor-core (tcgen05) backward for bf16 inputs, dk = dv = 64, chunks of
// C = 128 tokens: causal (two sweeps), and non-causal (passes A and B below).
//
// Gradients of L = sum(dout * out) by cumulative sums, with no per-token
// state stored ("Transformers are RNNs" review, section "그래디언트 계산 —
// 선형 시간·상수 메모리" names the method; its formulas did not survive on
// the page and are derived here from the forward definition). With
// g_t = dout_t, D_t = phi(q_t).z_t + eps (inclusive z_t) and
// o_t = S_t^T phi(q_t) / D_t:
//   a_t = g_t / D_t,  b_t = -(g_t . o_t) / D_t
//   dphi(q_t) = S_t a_t + b_t z_t
//   R_j = sum_{t>=j} phi(q_t) a_t^T,  r_j = sum_{t>=j} b_t phi(q_t)
//   dphi(k_j) = R_j v_j + r_j,  dv_j = R_j^T phi(k_j)
//   dq = dphi(q) * phi'(q),  dk = dphi(k) * phi'(k),  phi'(x) = min(phi(x), 1)
//
// dq is ill-conditioned in the feature values: dphi(q_t) = sum_j phi(k_j)
// ((v_j - o_t) . a_t), and phi(k) = 1 + psi(k) has a common part (the 1)
// whose terms cancel almost exactly, leaving a sum some 10-50 times smaller
// than its terms for inputs of unit scale. Rounding phi(k) to bf16 (2^-9 of
// the 1) would therefore cost percents of dq. Sweep 1 and pass A split phi(k)
// = 1 + psi(k): the tensor cores see only psi(k) (bf16 rounding relative to
// psi, which is small), and the parts that carry the 1 are exact fp32
// scalars per row. With s_t = sum_i phi(q_t)_i, V_t = sum_{j<=t} v_j and n_t =
// t + 1 (tokens up to t):
//   D_t = s_t n_t + phi(q_t).z_psi,t + eps
//   a_t . O_t = s_t a_t . V_t + a_t . O_psi,t,  O_psi,t = S_psi,t^T phi(q_t)
//   dphi(q_t) = c_t 1 + S_psi,t a_t + b_t z_psi,t,  c_t = a_t . V_t + n_t b_t
// where S_psi, z_psi sum psi(k) in place of phi(k), and a_t is the bf16 a of
// the MMAs in every term (b_t = -a_t . O_t / D_t is formed from it too).
//
// Sweep 1 (forward through each segment, from the segment's centred prefix
// S_psi, z_psi and the sum of v before it; the state is held transposed):
//   P    = phi(Q) psi(K)^T, masked j <= t           MMA (both K-major)
//   O    = phi(Q) S_psi,prev + P V                  MMA, MMA (P from TMEM)
//   S_psi^T += V^T psi(K)                           MMA
//   den  = s n + phi(Q) z_psi,prev + P 1 + eps;  a = g / den (bf16)
//   dP   = a V^T;  rho = (dP 1) masked j <= t      MMA, CUDA cores
//   b = -(s (a . V_prev + rho) + a . O) / den;  c = a . V_prev + rho + n b
//   dP'  = (dP + b) masked j <= t                   CUDA cores
//   dQ   = a S_psi,prev^T + dP' psi(K) + b z_psi,prev + c    MMA, MMA, epilogue
//   R   += phi(Q)^T a;  r += phi(Q)^T b             MMA, CUDA cores
// writing dq, (den, b) per token and the segment's (R, r) sums.
// Sweep 2 (backward through each segment, from the suffix R, r after it):
//   P^T  = phi(K) phi(Q)^T, masked t >= j           MMA
//   dP^T = V a^T;  dP^T' = (dP^T + b_t) masked      MMA, CUDA cores
//   dK   = V R_after^T + dP^T' phi(Q) + r_after     MMA, MMA, epilogue
//   dV   = phi(K) R_after + P^T' a                  MMA, MMA
//   R   += phi(Q)^T a;  r += phi(Q)^T b
// Each segment starts from the sum of the other segments' records: sweep 1
// adds the state pass's records of the segments before it, sweep 2 adds
// sweep 1's (R, r) records of the segments after it. Sweep 1 is launched as a
// dependent of the state pass and sweep 2 of sweep 1, so each fills its
// pipeline before it waits for the records.
//
// Every wait is bounded; on a timeout the CTA sets the device status word,
// drains, frees its tensor memory and exits. Barriers that a consumer may
// reach more than one phase late are double-buffered by chunk parity.
#include "la_tc_common.cuh"

namespace la {

namespace {

using namespace sm100;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 16-byte chunk `ch` (features 8 ch .. 8 ch + 7) of row r of a [C][D] tile
// stored as 64-feature SW128 boxes.
__device__ __forceinline__ uint4 ld_chunk(const uint8_t* tile, int r, int ch) {
  return *reinterpret_cast<const uint4*>(tile + (ch >> 3) * BOX + sw128(r, ch & 7));
}
__device__ __forceinline__ void st_chunk(uint8_t* tile, int r, int ch, uint4 v) {
  *reinterpret_cast<uint4*>(tile + (ch >> 3) * BOX + sw128(r, ch & 7)) = v;
}

// Causal mask of one 128-column fp32 row in tensor memory (row r = 32 q +
// lane of the chunk), packed to bf16 into the row's first 64 columns. kLower
// keeps columns j <= r (query rows against key columns), otherwise j >= r (key
// rows against query columns). Kept entries get `add_row` added, and with
// kColAdd also add_col[j]. Returns the sum of the kept fp32 entries.
template <bool kLower, bool kColAdd>
__device__ __forceinline__ float mask_pack_row(uint32_t taddr, int q, int lane, float add_row, const float* add_col) {
  float sum = 0.f;
#pragma unroll 1
  for (int p = 0; p < 4; ++p) {
    uint32_t pk[16];
    const bool live = kLower ? (p <= q) : (p >= q);
    if (live) {
      uint32_t v[32];
      tmem_ld32(taddr + 32 * p, v);
      float cb[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) cb[j] = 0.f;
      if (kColAdd) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 f = reinterpret_cast<const float4*>(add_col + 32 * p)[j];
          cb[4 * j] = f.x; cb[4 * j + 1] = f.y; cb[4 * j + 2] = f.z; cb[4 * j + 3] = f.w;
        }
      }
      tmem_ld_wait();
      if (p != q) {
        // a piece wholly on the kept side of the diagonal
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float x0 = __uint_as_float(v[2 * j]) + add_row + cb[2 * j];
          const float x1 = __uint_as_float(v[2 * j + 1]) + add_row + cb[2 * j + 1];
          sum += x0 + x1;
          pk[j] = pack_bf16x2(x0, x1);
        }
      } else {
        const int lo = kLower ? 0 : lane;       // kept columns [lo, hi)
        const int hi = kLower ? lane + 1 : 32;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int e0 = 2 * j, e1 = 2 * j + 1;
          const float x0 = (e0 >= lo && e0 < hi) ? __uint_as_float(v[e0]) + add_row + cb[e0] : 0.f;
          const float x1 = (e1 >= lo && e1 < hi) ? __uint_as_float(v[e1]) + add_row + cb[e1] : 0.f;
          sum += x0 + x1;
          pk[j] = pack_bf16x2(x0, x1);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[j] = 0u;
    }
    tmem_st16(taddr + 16 * p, pk);
  }
  return sum;
}

// phi(q_r) . z for row r of the phi-transformed Q tile (bf16) and fp32 z.
template <int D>
__device__ __forceinline__ float phiq_dot(const uint8_t* qtile, int r, const float* z) {
  float dot = 0.f;
#pragma unroll 2
  for (int ch = 0; ch < D / 8; ++ch) {
    const uint4 w = ld_chunk(qtile, r, ch);
    const uint32_t* pw = reinterpret_cast<const uint32_t*>(&w);
    const float4 z0 = *reinterpret_cast<const float4*>(z + 8 * ch);
    const float4 z1 = *reinterpret_cast<const float4*>(z + 8 * ch + 4);
    dot = fmaf(bf_lo(pw[0]), z0.x, dot);
    dot = fmaf(bf_hi(pw[0]), z0.y, dot);
    dot = fmaf(bf_lo(pw[1]), z0.z, dot);
    dot = fmaf(bf_hi(pw[1]), z0.w, dot);
    dot = fmaf(bf_lo(pw[2]), z1.x, dot);
    dot = fmaf(bf_hi(pw[2]), z1.y, dot);
    dot = fmaf(bf_lo(pw[3]), z1.z, dot);
    dot = fmaf(bf_hi(pw[3]), z1.w, dot);
  }
  return dot;
}

// As phiq_dot, also returning the row sum of phi(q_r) in *rs.
template <int D>
__device__ __forceinline__ float phiq_dot_sum(const uint8_t* qtile, int r, const float* z, float* rs) {
  float dot = 0.f, sum = 0.f;
#pragma unroll 2
  for (int ch = 0; ch < D / 8; ++ch) {
    const uint4 w = ld_chunk(qtile, r, ch);
    const uint32_t* pw = reinterpret_cast<const uint32_t*>(&w);
    const float4 z0 = *reinterpret_cast<const float4*>(z + 8 * ch);
    const float4 z1 = *reinterpret_cast<const float4*>(z + 8 * ch + 4);
    const float f[8] = {bf_lo(pw[0]), bf_hi(pw[0]), bf_lo(pw[1]), bf_hi(pw[1]),
                        bf_lo(pw[2]), bf_hi(pw[2]), bf_lo(pw[3]), bf_hi(pw[3])};
    const float zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      dot = fmaf(f[e], zz[e], dot);
      sum += f[e];
    }
  }
  *rs = sum;
  return dot;
}

// Row pass of the centred gradient: with the centred numerator row O_psi
// (fp32, tensor memory) and the upstream-gradient row g_r (bf16, G tile),
// overwrite g_r in place with a_r = g_r * inv_den rounded to bf16 (nearest)
// and return beta1 = a_r . O_psi, with beta0 = a_r . vsum in *beta0. Both
// dot products take the rounded a_r that the MMAs read, so that every term
// of the gradient is formed from the same a.
template <int D>
__device__ __forceinline__ float grad_row_pass_centred(uint32_t taddr, uint8_t* gtile, int r, float inv_den,
                                                       const float* vsum, float* beta0) {
  float b1 = 0.f, b0 = 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(taddr + c0, v);
    uint4 gw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) gw[j] = ld_chunk(gtile, r, c0 / 8 + j);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(&gw[j]);
      const float4 s0 = *reinterpret_cast<const float4*>(vsum + c0 + 8 * j);
      const float4 s1 = *reinterpret_cast<const float4*>(vsum + c0 + 8 * j + 4);
      const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      uint4 o;
      uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        po[h] = pack_bf16x2(bf_lo(pw[h]) * inv_den, bf_hi(pw[h]) * inv_den);
        const float a0 = bf_lo(po[h]), a1 = bf_hi(po[h]);
        b1 = fmaf(a0, __uint_as_float(v[8 * j + 2 * h]), b1);
        b1 = fmaf(a1, __uint_as_float(v[8 * j + 2 * h + 1]), b1);
        b0 = fmaf(a0, sv[2 * h], b0);
        b0 = fmaf(a1, sv[2 * h + 1], b0);
      }
      st_chunk(gtile, r, c0 / 8 + j, o);
    }
  }
  *beta0 = b0;
  return b1;
}

// The masked constant row [x for j <= r, 0 for j > r] (r = 32 q + lane) as
// 64 packed bf16 columns at tensor-memory address `taddr`.
__device__ __forceinline__ void store_lower_block(uint32_t taddr, int q, int lane, float x) {
  const uint32_t xx = pack_bf16x2(x, x), x0 = pack_bf16x2(x, 0.f);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      // columns 2j, 2j + 1 of piece p
      const int c0 = 2 * j;
      w[j] = p < q ? xx : p > q ? 0u : (c0 + 1 <= lane ? xx : c0 <= lane ? x0 : 0u);
    }
    tmem_st16(taddr + 16 * p, w);
  }
}

// Row pass of sweep 1: with the numerator row O_r (fp32, tensor memory) and
// the upstream-gradient row g_r (bf16, G tile), return beta = g_r . O_r and
// overwrite g_r in place with a_r = g_r * inv_den (bf16, nearest).
template <int D>
__device__ __forceinline__ float grad_row_pass(uint32_t taddr, uint8_t* gtile, int r, float inv_den) {
  float beta = 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(taddr + c0, v);
    uint4 gw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) gw[j] = ld_chunk(gtile, r, c0 / 8 + j);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(&gw[j]);
      uint4 o;
      uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float g0 = bf_lo(pw[h]), g1 = bf_hi(pw[h]);
        beta = fmaf(g0, __uint_as_float(v[8 * j + 2 * h]), beta);
        beta = fmaf(g1, __uint_as_float(v[8 * j + 2 * h + 1]), beta);
        po[h] = pack_bf16x2(g0 * inv_den, g1 * inv_den);
      }
      st_chunk(gtile, r, c0 / 8 + j, o);
    }
  }
  return beta;
}

// Epilogue row of a gradient: x = acc (tensor memory) + add_s * add_v +
// add_c, times phi'(.) = min(phi, 1) read from row r of a phi-transformed
// tile, written in bf16 to row r of the swizzled output tile `otile` (stored
// later with TMA). add_v is an fp32 vector of D entries.
template <int D>
__device__ __forceinline__ void grad_epilogue(uint32_t taddr, const uint8_t* ftile, int r, float add_s,
                                              const float* add_v, uint8_t* otile, float add_c = 0.f) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(taddr + c0, v);
    uint4 fw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) fw[j] = ld_chunk(ftile, r, c0 / 8 + j);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(&fw[j]);
      const float4 a0 = *reinterpret_cast<const float4*>(add_v + c0 + 8 * j);
      const float4 a1 = *reinterpret_cast<const float4*>(add_v + c0 + 8 * j + 4);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      uint4 o;
      uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float x0 =
            (fmaf(add_s, av[2 * h], __uint_as_float(v[8 * j + 2 * h])) + add_c) * fminf(bf_lo(pw[h]), 1.f);
        const float x1 =
            (fmaf(add_s, av[2 * h + 1], __uint_as_float(v[8 * j + 2 * h + 1])) + add_c) * fminf(bf_hi(pw[h]), 1.f);
        po[h] = pack_bf16x2(x0, x1);
      }
      st_chunk(otile, r, c0 / 8 + j, o);
    }
  }
}

// An fp32 tensor-memory row (D columns) in bf16 to row r of a swizzled tile.
template <int D>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, uint8_t* otile, int r) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(taddr + c0, v);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 o;
      o.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
      o.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
      o.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
      o.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
      st_chunk(otile, r, c0 / 8 + j, o);
    }
  }
}

// ---------------------------------------------------------------------------
// Sweep 1
// ---------------------------------------------------------------------------
template <int D>
struct B1 {
  static_assert(D == 64, "the tensor-core backward is laid out for D = 64");
  static constexpr int NB = D / 64;
  static constexpr int TILE = NB * BOX;
  static constexpr int ST = 3;                        // stages of Q, K, S^T copy, V, G
  static constexpr int SBUF = NB * D * 128;           // bf16 copy of S_prev^T
  // stage layout: the S_prev^T copy follows the K tile, so that
  // [phi(K) ; S_prev^T] is one K-major operand of 128 + D rows
  static constexpr int OFF_K = TILE;
  static constexpr int OFF_SC = 2 * TILE;
  static constexpr int OFF_V = 2 * TILE + SBUF;
  static constexpr int OFF_G = 3 * TILE + SBUF;
  static constexpr int STAGE = 4 * TILE + SBUF;
  static constexpr int KSTEPS = D / 16;
  // tensor memory columns: two [P | O] pairs (P then dP in place, O then dQ)
  __host__ __device__ static constexpr uint32_t col_pd(int pb) { return pb * (128 + D); }
  __host__ __device__ static constexpr uint32_t col_oq(int pb) { return pb * (128 + D) + 128; }
  static constexpr uint32_t COL_S = 2 * (128 + D);    // D
  static constexpr uint32_t COL_R = COL_S + D;        // D
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_R + D <= TMEM_COLS, "tensor memory budget");
  // shared memory
  static constexpr int OFF_ZST = ST * STAGE;              // [ST][D] z_psi before each staged chunk
  static constexpr int OFF_VST = OFF_ZST + ST * D * 4;    // [ST][D] sum of v before each staged chunk
  static constexpr int OFF_ROW = OFF_VST + ST * D * 4;    // [ST][C] (s_t, a.V_prev, a.O_psi, den) per row
  static constexpr int OFF_BARR = OFF_ROW + ST * C * 16;  // [ST][C] b_t of each staged chunk
  static constexpr int OFF_BAR = OFF_BARR + ST * C * 4;
  static constexpr int NBAR = 3 * ST + 21;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
  static constexpr int THREADS = 576;
};

struct Bwd1Params {
  int N, P, seg_len, F;
  float eps;
  const float* ws_state;   // [BH][P*F][rec_words] centred state-pass sums of segments 0..P-2
  float* ws_rev;           // [BH][P][rec_words] segment sums (R, r), all but the first segment
  float* ws_tok;           // [BH][N][2] (den, b) per token
  __nv_bfloat16* dq;       // [BH][N][D]
  int* status;
};

// Warp roles (576 threads):
//   warps 0-3    group C: psi(K) in place (exact fp32, rounded), z_psi and the
//                sum of v
//   warps 4-7    group A: phi(Q) in place; bf16 copies of S_psi,prev; the r
//                sums; final (R, r) store
//   warps 8-11   group B: P mask/pack and row sums, den, a (row pass)
//   warps 12-15  group D: rho, b and c; dP' mask/pack, dq epilogue
//   warp 16      TMA producer (Q, K, V, G)
//   warp 17      TMEM allocator and MMA issuer
template <int D>
__global__ void __launch_bounds__(576, 1)
tc_bwd1_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
               const __grid_constant__ CUtensorMap map_dq, const Bwd1Params prm) {
  using G = B1<D>;
  constexpr int ST = G::ST;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  float* zst = reinterpret_cast<float*>(sm + G::OFF_ZST);
  float* vst = reinterpret_cast<float*>(sm + G::OFF_VST);
  float4* rowinfo = reinterpret_cast<float4*>(sm + G::OFF_ROW);
  float* barr = reinterpret_cast<float*>(sm + G::OFF_BARR);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + G::OFF_BAR);
  uint64_t* full = bars;                 // [ST]
  uint64_t* phi_done = bars + ST;        // [ST]
  uint64_t* empty = bars + 2 * ST;       // [ST]
  uint64_t* x = bars + 3 * ST;
  uint64_t* p_full = x;                  // [2]
  uint64_t* p_ready = x + 2;             // [2]
  uint64_t* o_full = x + 6;              // [2]
  uint64_t* a_ready = x + 8;             // [2]
  uint64_t* dp_full = x + 10;            // [2]
  uint64_t* dp_ready = x + 12;           // [2]
  uint64_t* dq_full = x + 14;            // [2]
  uint64_t* oq_empty = x + 16;           // [2]
  uint64_t* s_full = x + 18;
  uint64_t* s_ready = x + 19;
  uint64_t* mma_fin = x + 20;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + G::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + G::OFF_MISC + 4);
  // sweep 2 may start filling its pipeline while this grid runs
  griddep_launch_dependents();
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(prm.status);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / prm.P, seg = blockIdx.x % prm.P;
  const int tok0 = seg * prm.seg_len;
  const int tok_end = min(prm.N, tok0 + prm.seg_len);
  const int nchunks = (tok_end - tok0 + C - 1) / C;
  constexpr long long RW = rec_words<D>();
  const long long rec = ((long long)bh * prm.P + seg) * RW;

  if (tid == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&phi_done[i], 256);
      mbar_init(&empty[i], 1 + 128 + 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_ready[i], 128);
      mbar_init(&o_full[i], 1);
      mbar_init(&a_ready[i], 128);
      mbar_init(&dp_full[i], 1);
      mbar_init(&dp_ready[i], 128);
      mbar_init(&dq_full[i], 1);
      mbar_init(&oq_empty[i], 128);
    }
    mbar_init(s_full, 1);
    mbar_init(s_ready, 128);
    mbar_init(mma_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 17) {
    tmem_alloc(tmem_slot, G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 16) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      tma_prefetch_desc(&map_g);
      // dq of a chunk is staged in its stage's K region; it is stored here,
      // once the stage's consumers are done, before the stage is refilled
      auto store_dq = [&](int c) {
        uint8_t* stg = sm + (c % ST) * G::STAGE;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) tma_store_3d(&map_dq, stg + G::OFF_K + b * BOX, 64 * b, tok0 + c * C, bh);
        tma_store_commit();
        tma_store_wait_read<0>();
      };
      int issued = 0;
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % ST;
        if (c >= ST) {
          ok = mbar_wait(&empty[s], ((c / ST) - 1) & 1, abort_flag, kTimeoutNs);
          if (!ok) break;
          store_dq(c - ST);
        }
        uint8_t* stg = sm + s * G::STAGE;
        mbar_arrive_expect_tx(&full[s], 4 * G::TILE);
        const int y = tok0 + c * C;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) {
          tma_load_3d(stg + b * BOX, &map_q, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + G::OFF_K + b * BOX, &map_k, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + G::OFF_V + b * BOX, &map_v, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + G::OFF_G + b * BOX, &map_g, &full[s], 64 * b, y, bh);
        }
        issued = c + 1;
      }
      // the chunks still in the ring
      for (int c = max(0, issued - ST); c < issued && ok; ++c) {
        ok = mbar_wait(&empty[c % ST], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (ok) store_dq(c);
      }
      tma_store_wait<0>();
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_drain(&full[c % ST], (c / ST) & 1, kTimeoutNs);
    }
  } else if (warp == 17) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_qk = make_idesc_bf16(128, 128, false, false);  // dP = a V^T
      constexpr uint32_t id_qs = make_idesc_bf16(128, 128 + D, false, false);  // [P | O] = phiQ [phiK ; S_prev^T]^T
      constexpr uint32_t id_as = make_idesc_bf16(128, D, false, true);     // dQ = a S_prev^T (S^T copy MN-major)
      constexpr uint32_t id_tt = make_idesc_bf16(D, D, true, true);        // S^T += V^T phiK, R += phiQ^T a
      constexpr uint32_t id_pv = make_idesc_bf16(128, D, false, true);     // O += P V, dQ += [dP | b] [psiK ; psiK]
      // The four MMA groups of a chunk wait on different CUDA-core passes;
      // the issuer polls them and issues whichever is ready, the oldest
      // chunk first, so that the front MMAs of chunk c + 1 and its P V run
      // while chunk c's passes are still busy. Per chunk, in order:
      //   F  [P | O] = phiQ [psiK ; S_psi^T]^T and the state update   (phi/psi, S copy, buffers of c - 2 free)
      //   PV O += P V                                                (P packed)
      //   G  dP = a V^T, dQ = a S_psi^T, R += phiQ^T a               (a written)
      //   Q2 dQ += [dP | b] [psiK ; psiK]                            (dP and b packed)
      // F of chunk c needs Q2 of c - 2 issued (its P/dP buffer is then read
      // before F overwrites it: MMAs run in issue order).
      auto stage_addr = [&](int c) { return smem_u32(sm + (c % ST) * G::STAGE); };
      auto issue_f = [&](int c) {
        const int pb = c & 1;
        const uint32_t qa = stage_addr(c), ka = qa + G::OFF_K, va = qa + G::OFF_V;
        const uint32_t pd = tmem + G::col_pd(pb);
        // P and O = phiQ S_psi,prev share A = phiQ: one MMA over [psiK ; S_psi^T]
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(pd, make_sdesc(qa + off, 16, 1024, kSwizzle128B), make_sdesc(ka + off, 16, 1024, kSwizzle128B),
                 id_qs, k > 0);
        }
        tc_commit(&p_full[pb]);
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ss(tmem + G::COL_S, make_sdesc(va + k * 2048, BOX, 1024, kSwizzle128B),
                 make_sdesc(ka + k * 2048, BOX, 1024, kSwizzle128B), id_tt, 1);
        tc_commit(s_full);
      };
      auto issue_pv = [&](int c) {
        const int pb = c & 1;
        const uint32_t va = stage_addr(c) + G::OFF_V;
        const uint32_t pd = tmem + G::col_pd(pb), oq = tmem + G::col_oq(pb);
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ts(oq, pd + k * 8, make_sdesc(va + k * 2048, BOX, 1024, kSwizzle128B), id_pv, 1);
        tc_commit(&o_full[pb]);
      };
      auto issue_g = [&](int c) {
        const int pb = c & 1;
        const uint32_t qa = stage_addr(c), va = qa + G::OFF_V, ga = qa + G::OFF_G, sb = qa + G::OFF_SC;
        const uint32_t pd = tmem + G::col_pd(pb), oq = tmem + G::col_oq(pb);
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(pd, make_sdesc(ga + off, 16, 1024, kSwizzle128B), make_sdesc(va + off, 16, 1024, kSwizzle128B),
                 id_qk, k > 0);
        }
        tc_commit(&dp_full[pb]);
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k)
          mma_ss(oq, make_sdesc(ga + (k >> 2) * BOX + (k & 3) * 32, 16, 1024, kSwizzle128B),
                 make_sdesc(sb + k * 2048, D * 128, 1024, kSwizzle128B), id_as, k > 0);
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ss(tmem + G::COL_R, make_sdesc(qa + k * 2048, BOX, 1024, kSwizzle128B),
                 make_sdesc(ga + k * 2048, BOX, 1024, kSwizzle128B), id_tt, (c > 0 || k > 0) ? 1u : 0u);
      };
      auto issue_q2 = [&](int c) {
        const int pb = c & 1;
        const uint32_t ka = stage_addr(c) + G::OFF_K;
        const uint32_t pd = tmem + G::col_pd(pb), oq = tmem + G::col_oq(pb);
        // K = 256: the packed dP (columns 0..63) and the b block (64..127),
        // both against psiK
#pragma unroll
        for (int k = 0; k < 2 * C / 16; ++k)
          mma_ts(oq, pd + k * 8, make_sdesc(ka + (k & 7) * 2048, BOX, 1024, kSwizzle128B), id_pv, 1);
        tc_commit(&dq_full[pb]);
        tc_commit(&empty[c % ST]);
      };
      int nf = 0, npv = 0, ng = 0, nq = 0;   // next chunk of each MMA group
      bool ok = true;
      uint64_t t_last = globaltimer_ns();
      while (nq < nchunks) {
        bool issued = false;
        if (nq < ng && mbar_try_wait(&dp_ready[nq & 1], (nq >> 1) & 1)) {
          tc_fence_after();
          issue_q2(nq++);
          issued = true;
        } else if (ng < npv && mbar_try_wait(&a_ready[ng & 1], (ng >> 1) & 1)) {
          tc_fence_after();
          issue_g(ng++);
          issued = true;
        } else if (npv < nf && mbar_try_wait(&p_ready[npv & 1], (npv >> 1) & 1)) {
          tc_fence_after();
          issue_pv(npv++);
          issued = true;
        } else if (nf < nchunks && nf <= nq + 1 && mbar_try_wait(&phi_done[nf % ST], (nf / ST) & 1) &&
                   mbar_try_wait(s_ready, nf & 1) &&
                   (nf < 2 || (mbar_try_wait(&dq_full[nf & 1], ((nf >> 1) - 1) & 1) &&
                               mbar_try_wait(&oq_empty[nf & 1], ((nf >> 1) - 1) & 1)))) {
          tc_fence_after();
          issue_f(nf++);
          issued = true;
        }
        if (issued) {
          t_last = globaltimer_ns();
        } else if (*abort_flag || globaltimer_ns() - t_last > kTimeoutNs) {
          *abort_flag = 1;
          ok = false;
          break;
        }
      }
      (void)ok;
      tc_commit(mma_fin);
      mbar_drain(mma_fin, 0, kTimeoutNs);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- group A: phi(Q), S_prev copies, the r sums, R ----------------
    using X = ExactLayout<D, 128>;
    const int t = tid - 128;
    const int q = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    const int fc = X::FCW * (t >> 5) + (lane % X::FCW);
    float racc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) racc[e] = 0.f;
    griddep_wait();
    // the centred prefix S_psi^T (the held state stays centred)
    sum_states_to_tmem<D>(prm.ws_state + (long long)bh * prm.P * prm.F * RW, RW, 0, seg * prm.F, lane_addr,
                          G::COL_S, row);
    bool ok = true;
    for (int c = 0; c <= nchunks && ok; ++c) {
      if (c < nchunks) {
        const int s = c % ST;
        ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        phi_tile_bf16<D, 128>(sm + s * G::STAGE, t);
        fence_proxy_async_smem();
        mbar_arrive(&phi_done[s]);
        if (c > 0) ok = mbar_wait(s_full, (c - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        copy_state_to_smem<D>(lane_addr + G::COL_S, sm + s * G::STAGE + G::OFF_SC, row);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(s_ready);
      }
      if (c >= 1) {
        // r += sum_t b_t phi(q_t) over the previous chunk (b from group D);
        // here rather than in group C, so that the psi(K) passes never wait
        // for a chunk's dP pack
        const int cp = c - 1, sp = cp % ST;
        ok = mbar_wait(&dp_ready[cp & 1], (cp >> 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        wcolsum_tile<D, 128>(sm + sp * G::STAGE, barr + sp * C, t, racc);
        mbar_arrive(&empty[sp]);
      }
    }
    reduce_row_groups<D, 128>(racc);
    if (ok && lane < X::FCW && seg > 0) {
      float4* rd = reinterpret_cast<float4*>(prm.ws_rev + rec + D * D + 8 * fc);
      rd[0] = make_float4(racc[0], racc[1], racc[2], racc[3]);
      rd[1] = make_float4(racc[4], racc[5], racc[6], racc[7]);
    }
    // the first segment's (R, r) sums are never read
    if (ok && seg > 0) ok = mbar_wait(mma_fin, 0, abort_flag, kTimeoutNs);
    if (ok && seg > 0) {
      tc_fence_after();
      store_state_from_tmem<D>(prm.ws_rev + rec, lane_addr, G::COL_R, row);
    }
  } else if (warp >= 8 && warp < 12) {
    // ---------------- group B: P, den, a and b ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST, pb = c & 1;
      // phi(q_r) . z_psi,prev and s_r need only the phi tiles: formed while
      // the MMAs of the chunk run, before P is ready
      ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      float srow;
      const float qz = phiq_dot_sum<D>(sm + s * G::STAGE, r, zst + s * D, &srow);
      ok = mbar_wait(&p_full[pb], (c >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      const float rowsum = mask_pack_row<true, false>(lane_addr + G::col_pd(pb), q, lane, 0.f, nullptr);
      // tokens up to and including this row: the 1 of every phi(k_j) in z_t
      const float n_t = (float)(tok0 + c * C + r + 1);
      const float den = fmaf(srow, n_t, rowsum + qz) + prm.eps;
      const float inv_den = 1.f / den;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_ready[pb]);
      ok = mbar_wait(&o_full[pb], (c >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      float beta0;
      const float beta1 = grad_row_pass_centred<D>(lane_addr + G::col_oq(pb), sm + s * G::STAGE + G::OFF_G, r,
                                                   inv_den, vst + s * D, &beta0);
      rowinfo[s * C + r] = make_float4(srow, beta0, beta1, den);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&a_ready[pb]);
    }
  } else if (warp >= 12 && warp < 16) {
    // ---------------- group D: dP', dq ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    float2* tokp = reinterpret_cast<float2*>(prm.ws_tok) + (long long)bh * prm.N;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST, pb = c & 1;
      ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs) &&
           mbar_wait(&dp_full[pb], (c >> 1) & 1, abort_flag, kTimeoutNs) &&
           mbar_wait(&a_ready[pb], (c >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      // the masked dP row packed to bf16 (columns 0..63) with its fp32 sum
      // rho = a . (v_j summed over j <= t in the chunk); then b, c and the
      // masked b block (columns 64..127): dP' = dP + b enters dQ as
      // [dP | b] [psiK ; psiK]. c and b depend on rho only through small
      // terms (c = (Y a.V_t - n a.O_psi) / den with Y = den - s n), so the
      // two roundings cost no accuracy.
      const float rho = mask_pack_row<true, false>(lane_addr + G::col_pd(pb), q, lane, 0.f, nullptr);
      const float4 ri = rowinfo[s * C + r];     // (s_t, a.V_prev, a.O_psi, den)
      const int tok = tok0 + c * C + r;
      const float av = ri.y + rho;              // a . V_t
      const float b = -fmaf(ri.x, av, ri.z) / ri.w;
      const float cterm = fmaf((float)(tok + 1), b, av);
      barr[s * C + r] = b;
      if (tok < tok_end) tokp[tok] = make_float2(ri.w, b);
      store_lower_block(lane_addr + G::col_pd(pb) + 64, q, lane, b);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&dp_ready[pb]);
      ok = mbar_wait(&dq_full[pb], (c >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      // dq staged in the chunk's K region (dead once dQ += dP' psiK is done);
      // the TMA producer stores it before refilling the stage
      grad_epilogue<D>(lane_addr + G::col_oq(pb), sm + s * G::STAGE, r, b, zst + s * D,
                       sm + s * G::STAGE + G::OFF_K, cterm);
      tc_fence_before();
      mbar_arrive(&oq_empty[pb]);
      fence_proxy_async_smem();
      mbar_arrive(&empty[s]);
    }
  } else {
    // ---------------- group C: psi(K), z_psi and the sum of v ----------------
    using X = ExactLayout<D, 128>;
    const int t = tid;
    const int fc = X::FCW * (t >> 5) + (lane % X::FCW);
    const bool owner = lane < X::FCW;
    float zrun[8], vrun[8];
    griddep_wait();
    // z_psi and the sum of v before the segment, from the centred records
    sum_vectors8<D>(prm.ws_state + (long long)bh * prm.P * prm.F * RW, RW, 0, seg * prm.F, 8 * fc, zrun);
    sum_vectors8<D>(prm.ws_state + (long long)bh * prm.P * prm.F * RW, RW, 0, seg * prm.F, D + 8 * fc, vrun);
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      const int n_valid = min(C, tok_end - (tok0 + c * C));
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      float colsum[8], vcol[8];
      phi_tile_exact<D, 128, true, true, false, true>(sm + s * G::STAGE + G::OFF_K, t, n_valid, colsum);
      fence_proxy_async_smem();
#pragma unroll
      for (int e = 0; e < 8; ++e) vcol[e] = 0.f;
      colsum_tile<D, 128>(sm + s * G::STAGE + G::OFF_V, t, n_valid, vcol);
      reduce_row_groups<D, 128>(vcol);
      if (owner) {
        float4* zd = reinterpret_cast<float4*>(zst + s * D + 8 * fc);
        zd[0] = make_float4(zrun[0], zrun[1], zrun[2], zrun[3]);
        zd[1] = make_float4(zrun[4], zrun[5], zrun[6], zrun[7]);
        float4* vd = reinterpret_cast<float4*>(vst + s * D + 8 * fc);
        vd[0] = make_float4(vrun[0], vrun[1], vrun[2], vrun[3]);
        vd[1] = make_float4(vrun[4], vrun[5], vrun[6], vrun[7]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          zrun[e] += colsum[e];
          vrun[e] += vcol[e];
        }
      }
      mbar_arrive(&phi_done[s]);
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  // after the barrier: a warp that gave up late is seen too
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  if (warp == 17) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Sweep 2
// ---------------------------------------------------------------------------
template <int D>
struct B2 {
  static_assert(D == 64, "the tensor-core backward is laid out for D = 64");
  static constexpr int NB = D / 64;
  static constexpr int TILE = NB * BOX;
  static constexpr int ST = 3;
  static constexpr int RBUF = NB * D * 128;           // bf16 copy of R_after
  // stage: Q, K, V, G (becomes a in place), then the R_after copy right after
  // the a tile, so that [a ; R_after] is one K-major operand of 128 + D rows
  static constexpr int OFF_R = 4 * TILE;
  static constexpr int STAGE = OFF_R + RBUF;
  static constexpr int KSTEPS = D / 16;
  static constexpr uint32_t COL_PT = 0;               // 128
  static constexpr uint32_t COL_DPT = 128;            // 128, followed by dK: [dP^T | dK] from one MMA
  static constexpr uint32_t COL_DK = 256;             // D
  static constexpr uint32_t COL_DV = COL_DK + D;      // D
  static constexpr uint32_t COL_R = COL_DV + D;       // D
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_R + D <= TMEM_COLS, "tensor memory budget");
  static_assert(COL_DK == COL_DPT + 128, "dK must follow dP^T");
  static constexpr int OFF_RVEC = ST * STAGE;             // [2][D] r_after
  static constexpr int OFF_BARR = OFF_RVEC + 2 * D * 4;   // [ST][C] b_t
  static constexpr int OFF_BAR = OFF_BARR + ST * C * 4;
  static constexpr int NBAR = 3 * ST + 12;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
  static constexpr int THREADS = 448;
};

struct Bwd2Params {
  int N, P, seg_len;
  const float* ws_rev;     // [BH][P][rec_words] segment sums (R, r), all but the first segment
  const float* ws_tok;     // [BH][N][2] (den, b)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
};

// Warp roles (448 threads); chunks run from the segment's end to its start:
//   warps 0-3    group C: phi(K) in place; a = g / den in place; b_t
//   warps 4-7    group A: phi(Q) in place; R_after copies; r_after sums
//   warps 8-11   group D: P^T' and dP^T' mask/pack; dk, dv epilogue
//   warp 12      TMA producer
//   warp 13      TMEM allocator and MMA issuer
template <int D>
__global__ void __launch_bounds__(448, 1)
tc_bwd2_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
               const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
               const Bwd2Params prm) {
  using G = B2<D>;
  constexpr int ST = G::ST;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  float* rvec = reinterpret_cast<float*>(sm + G::OFF_RVEC);
  float* barr = reinterpret_cast<float*>(sm + G::OFF_BARR);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + G::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* prep_done = bars + ST;
  uint64_t* empty = bars + 2 * ST;
  uint64_t* x = bars + 3 * ST;
  uint64_t* pt_full = x;
  uint64_t* dpt_full = x + 1;
  uint64_t* pt_ready = x + 2;
  uint64_t* dpt_ready = x + 3;
  uint64_t* rb_ready = x + 4;     // [2]
  uint64_t* r_full = x + 6;
  uint64_t* kv_full = x + 7;
  uint64_t* kv_empty = x + 8;     // [2]
  uint64_t* mma_fin = x + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + G::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + G::OFF_MISC + 4);
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(prm.status);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / prm.P, seg = blockIdx.x % prm.P;
  const int tok0 = seg * prm.seg_len;
  const int tok_end = min(prm.N, tok0 + prm.seg_len);
  const int nchunks = (tok_end - tok0 + C - 1) / C;

  if (tid == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&prep_done[i], 256);
      mbar_init(&empty[i], 1 + 128 + 128);
    }
    mbar_init(pt_full, 1);
    mbar_init(dpt_full, 1);
    mbar_init(pt_ready, 128);
    mbar_init(dpt_ready, 128);
    mbar_init(&rb_ready[0], 128);
    mbar_init(&rb_ready[1], 128);
    mbar_init(r_full, 1);
    mbar_init(kv_full, 1);
    mbar_init(&kv_empty[0], 128);
    mbar_init(&kv_empty[1], 128);
    mbar_init(mma_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
    // ---------------- TMA producer (last chunk first) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      tma_prefetch_desc(&map_g);
      // dk and dv of iteration i are staged in its stage's V and a tiles;
      // they are stored here, once the stage's consumers are done
      auto store_dkv = [&](int i) {
        uint8_t* stg = sm + (i % ST) * G::STAGE;
        const int y = tok0 + (nchunks - 1 - i) * C;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) {
          tma_store_3d(&map_dk, stg + 2 * G::TILE + b * BOX, 64 * b, y, bh);
          tma_store_3d(&map_dv, stg + 3 * G::TILE + b * BOX, 64 * b, y, bh);
        }
        tma_store_commit();
        tma_store_wait_read<0>();
      };
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < nchunks; ++i) {
        const int s = i % ST;
        if (i >= ST) {
          ok = mbar_wait(&empty[s], ((i / ST) - 1) & 1, abort_flag, kTimeoutNs);
          if (!ok) break;
          store_dkv(i - ST);
        }
        uint8_t* stg = sm + s * G::STAGE;
        mbar_arrive_expect_tx(&full[s], 4 * G::TILE);
        const int y = tok0 + (nchunks - 1 - i) * C;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) {
          tma_load_3d(stg + b * BOX, &map_q, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + G::TILE + b * BOX, &map_k, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + 2 * G::TILE + b * BOX, &map_v, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + 3 * G::TILE + b * BOX, &map_g, &full[s], 64 * b, y, bh);
        }
        issued = i + 1;
      }
      // the chunks still in the ring
      for (int i = max(0, issued - ST); i < issued && ok; ++i) {
        ok = mbar_wait(&empty[i % ST], (i / ST) & 1, abort_flag, kTimeoutNs);
        if (ok) store_dkv(i);
      }
      tma_store_wait<0>();
      for (int i = max(0, issued - ST); i < issued; ++i)
        mbar_drain(&full[i % ST], (i / ST) & 1, kTimeoutNs);
    }
  } else if (warp == 13) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_kq = make_idesc_bf16(128, 128, false, false);  // P^T = phiK phiQ^T
      constexpr uint32_t id_vr = make_idesc_bf16(128, 128 + D, false, false);  // [dP^T | dK] = V [a ; R]^T
      constexpr uint32_t id_kr = make_idesc_bf16(128, D, false, true);     // dV = phiK R
      constexpr uint32_t id_tt = make_idesc_bf16(D, D, true, true);        // R += phiQ^T a
      constexpr uint32_t id_pv = make_idesc_bf16(128, D, false, true);     // dK += dP^T' phiQ, dV += P^T' a
      const uint32_t pt = tmem + G::COL_PT, dpt = tmem + G::COL_DPT;
      const uint32_t dkc = tmem + G::COL_DK, dvc = tmem + G::COL_DV;
      bool ok = true;
      for (int i = 0; i < nchunks && ok; ++i) {
        const int s = i % ST;
        const uint32_t qa = smem_u32(sm + s * G::STAGE);
        const uint32_t ka = qa + G::TILE, va = qa + 2 * G::TILE, ga = qa + 3 * G::TILE, rb = qa + G::OFF_R;
        ok = mbar_wait(&prep_done[s], (i / ST) & 1, abort_flag, kTimeoutNs);
        // the P^T / dP^T buffers are free once the previous chunk's MMAs are done
        if (ok && i >= 1) ok = mbar_wait(kv_full, (i - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(pt, make_sdesc(ka + off, 16, 1024, kSwizzle128B), make_sdesc(qa + off, 16, 1024, kSwizzle128B),
                 id_kq, k > 0);
        }
        tc_commit(pt_full);
        ok = mbar_wait(&rb_ready[i & 1], (i >> 1) & 1, abort_flag, kTimeoutNs);
        if (ok && i >= 1) ok = mbar_wait(&kv_empty[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        // dP^T = V a^T and dK = V R_after^T share A = V: one MMA over [a ; R_after]
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(dpt, make_sdesc(va + off, 16, 1024, kSwizzle128B), make_sdesc(ga + off, 16, 1024, kSwizzle128B),
                 id_vr, k > 0);
        }
        tc_commit(dpt_full);
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(dvc, make_sdesc(ka + off, 16, 1024, kSwizzle128B),
                 make_sdesc(rb + k * 2048, D * 128, 1024, kSwizzle128B), id_kr, k > 0);
        }
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ss(tmem + G::COL_R, make_sdesc(qa + k * 2048, BOX, 1024, kSwizzle128B),
                 make_sdesc(ga + k * 2048, BOX, 1024, kSwizzle128B), id_tt, 1);
        tc_commit(r_full);
        ok = mbar_wait(pt_ready, i & 1, abort_flag, kTimeoutNs) && mbar_wait(dpt_ready, i & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ts(dkc, dpt + k * 8, make_sdesc(qa + k * 2048, BOX, 1024, kSwizzle128B), id_pv, 1);
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ts(dvc, pt + k * 8, make_sdesc(ga + k * 2048, BOX, 1024, kSwizzle128B), id_pv, 1);
        tc_commit(kv_full);
        tc_commit(&empty[s]);
      }
      tc_commit(mma_fin);
      mbar_drain(mma_fin, 0, kTimeoutNs);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- group A: phi(Q), R_after copies, r_after ----------------
    using X = ExactLayout<D, 128>;
    const int t = tid - 128;
    const int q = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    const int fc = X::FCW * (t >> 5) + (lane % X::FCW);
    const bool owner = lane < X::FCW;
    // R_after, r_after of the segment: the sums of the segments after it
    const float* recs = prm.ws_rev + (long long)bh * prm.P * rec_words<D>();
    float rrun[8];
    griddep_wait();
    sum_states_to_tmem<D>(recs, rec_words<D>(), seg + 1, prm.P, lane_addr, G::COL_R, row);
    sum_vectors8<D>(recs, rec_words<D>(), seg + 1, prm.P, 8 * fc, rrun);
    bool ok = true;
    for (int i = 0; i < nchunks && ok; ++i) {
      const int s = i % ST;
      ok = mbar_wait(&full[s], (i / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      phi_tile_bf16<D, 128>(sm + s * G::STAGE, t);
      fence_proxy_async_smem();
      mbar_arrive(&prep_done[s]);
      // R_after of chunk i: R after the updates of every later chunk
      if (i > 0) ok = mbar_wait(r_full, (i - 1) & 1, abort_flag, kTimeoutNs);
      // r_after of chunk i goes where chunk i - 2's epilogue read it
      if (ok && i >= 2) ok = mbar_wait(&kv_empty[i & 1], ((i - 2) >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      copy_state_to_smem<D>(lane_addr + G::COL_R, sm + s * G::STAGE + G::OFF_R, row);
      if (owner) {
        float4* rd = reinterpret_cast<float4*>(rvec + (i & 1) * D + 8 * fc);
        rd[0] = make_float4(rrun[0], rrun[1], rrun[2], rrun[3]);
        rd[1] = make_float4(rrun[4], rrun[5], rrun[6], rrun[7]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&rb_ready[i & 1]);
      // r += sum_t b_t phi(q_t) over this chunk (b from group C)
      ok = mbar_wait(&prep_done[s], (i / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      float racc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) racc[e] = 0.f;
      wcolsum_tile<D, 128>(sm + s * G::STAGE, barr + s * C, t, racc);
      reduce_row_groups<D, 128>(racc);
#pragma unroll
      for (int e = 0; e < 8; ++e) rrun[e] += racc[e];
      mbar_arrive(&empty[s]);
    }
  } else if (warp >= 8 && warp < 12) {
    // ---------------- group D: P^T', dP^T', dk, dv ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;            // key row j of the chunk
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    bool ok = true;
    for (int i = 0; i < nchunks && ok; ++i) {
      const int s = i % ST;
      ok = mbar_wait(&prep_done[s], (i / ST) & 1, abort_flag, kTimeoutNs) &&
           mbar_wait(&rb_ready[i & 1], (i >> 1) & 1, abort_flag, kTimeoutNs) &&
           mbar_wait(pt_full, i & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      mask_pack_row<false, false>(lane_addr + G::COL_PT, q, lane, 0.f, nullptr);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(pt_ready);
      ok = mbar_wait(dpt_full, i & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      mask_pack_row<false, true>(lane_addr + G::COL_DPT, q, lane, 0.f, barr + s * C);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(dpt_ready);
      ok = mbar_wait(kv_full, i & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      // dk and dv staged in the chunk's V and a tiles (dead once its MMAs are
      // done); the TMA producer stores them before refilling the stage
      uint8_t* stg = sm + s * G::STAGE;
      grad_epilogue<D>(lane_addr + G::COL_DK, stg + G::TILE, r, 1.f, rvec + (i & 1) * D, stg + 2 * G::TILE);
      store_row_bf16<D>(lane_addr + G::COL_DV, stg + 3 * G::TILE, r);
      tc_fence_before();
      mbar_arrive(&kv_empty[i & 1]);
      fence_proxy_async_smem();
      mbar_arrive(&empty[s]);
    }
  } else {
    // ---------------- group C: phi(K), a = g / den, b ----------------
    const int t = tid;                      // chunk row for the a scaling
    const float2* tokp = reinterpret_cast<const float2*>(prm.ws_tok) + (long long)bh * prm.N;
    griddep_wait();
    bool ok = true;
    for (int i = 0; i < nchunks && ok; ++i) {
      const int s = i % ST;
      const int y = tok0 + (nchunks - 1 - i) * C;
      const bool valid = y + t < tok_end;
      const float2 db = valid ? tokp[y + t] : make_float2(1.f, 0.f);
      ok = mbar_wait(&full[s], (i / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      uint8_t* stg = sm + s * G::STAGE;
      phi_tile_bf16<D, 128>(stg + G::TILE, t);
      const float inv = valid ? 1.f / db.x : 0.f;
      uint8_t* gt = stg + 3 * G::TILE;
#pragma unroll 2
      for (int ch = 0; ch < D / 8; ++ch) {
        const uint4 w = ld_chunk(gt, t, ch);
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(&w);
        uint4 o;
        o.x = pack_bf16x2(bf_lo(pw[0]) * inv, bf_hi(pw[0]) * inv);
        o.y = pack_bf16x2(bf_lo(pw[1]) * inv, bf_hi(pw[1]) * inv);
        o.z = pack_bf16x2(bf_lo(pw[2]) * inv, bf_hi(pw[2]) * inv);
        o.w = pack_bf16x2(bf_lo(pw[3]) * inv, bf_hi(pw[3]) * inv);
        st_chunk(gt, t, ch, o);
      }
      barr[s * C + t] = valid ? db.y : 0.f;
      fence_proxy_async_smem();
      mbar_arrive(&prep_done[s]);
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  // after the barrier: a warp that gave up late is seen too
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Non-causal backward (every query reads S_N, z_N; every key sees R_0, r_0):
//   D_t = phi(q_t).z_N + eps,  a_t = g_t / D_t,  b_t = -(g_t . o_t) / D_t,
//   dphi(q_t) = S_N a_t + b_t z_N,
//   R_0 = sum_t phi(q_t) a_t^T,  r_0 = sum_t b_t phi(q_t),
//   dphi(k_j) = R_0 v_j + r_0,  dv_j = R_0^T phi(k_j)
// (the non-causal case of the gradient above: S_t -> S_N, R_j -> R_0).
// Three launches: the forward's state pass over all segments (S_N, z_N
// records), pass A per segment (dq and the segment's (R, r) record), pass B
// per segment (dk, dv from the sum of all (R, r) records). No masks: each
// chunk is a dense product with the totals.
// ---------------------------------------------------------------------------
template <int D>
struct NA {
  static_assert(D == 64, "the tensor-core backward is laid out for D = 64");
  static constexpr int TILE = BOX;
  // stages of Q, G: a stage lives from its load through the row pass, the
  // MMAs, the dq epilogue and the store (~5 us), so six keep the loads going
  static constexpr int ST = 6;
  static constexpr int OFF_G = TILE;
  static constexpr int STAGE = 2 * TILE;
  // bf16 [S_psi,N^T ; z_hi ; z_lo ; 1 ; 0] (D + 16 rows): O_psi, phi(q).z_psi
  // and the row sum s_t of phi(q) from one MMA
  static constexpr int NO = D + 16;
  static constexpr uint32_t G_NO = NO;
  static constexpr int OFF_SBUF = ST * STAGE;
  static constexpr int OFF_ZN = OFF_SBUF + NO * 128;  // [D] z_psi,N (fp32)
  static constexpr int OFF_VN = OFF_ZN + D * 4;       // [D] sum of all v (fp32)
  static constexpr int OFF_BARR = OFF_VN + D * 4;     // [ST][C] b_t
  static constexpr int OFF_CARR = OFF_BARR + ST * C * 4;  // [ST][C] c_t
  static constexpr int OFF_BAR = OFF_CARR + ST * C * 4;
  static constexpr int NBAR = 6 * ST + 8 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
  static constexpr uint32_t COL_S = 0;                // S_N^T (M = D layout), start only
  static constexpr uint32_t COL_R = 64;               // R (M = D layout)
  // [O | den parts] of a chunk (free once its row pass is done) and dQ of a
  // chunk (free once its epilogue is done), each double-buffered
  __host__ __device__ static constexpr uint32_t col_o(int ob) { return 128 + G_NO * ob; }
  __host__ __device__ static constexpr uint32_t col_dq(int ob) { return 128 + 2 * G_NO + D * ob; }
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(col_dq(1) + D <= TMEM_COLS, "tensor memory budget");
  static constexpr int THREADS = 448;
};

struct NcBwdParams {
  int N, P, seg_len, F;
  float eps;
  const float* ws_state;   // [BH][P*F][rec_words] centred sums of every part (pass A reads)
  float* ws_rev;           // [BH][P][rec_words] (R, r) of each segment (A writes, B reads)
  int* status;
};

// Pass A (448 threads). Warps 0-3: phi(Q), the centred S_psi,N / z_psi,N sums
// and copy, the r sums and the (R, r) record; warps 4-7: the row pass (a, b,
// c) from [O_psi | phi(q).z_psi | s]; warps 8-11: the dq epilogue; warp 12
// TMA (Q, G in; dq out from the dead G tile); warp 13 TMEM and MMA. In the
// centred form of sweep 1 with every token before every query (n_t = N,
// V_t = the sum of all v, no intra-chunk term):
//   D_t = s_t N + phi(q_t).z_psi,N + eps,  a_t = g_t / D_t (bf16)
//   b_t = -(s_t a_t . V_N + a_t . O_psi,t) / D_t,  c_t = a_t . V_N + N b_t
//   dphi(q_t) = S_psi,N a_t + b_t z_psi,N + c_t
template <int D>
__global__ void __launch_bounds__(448, 1)
tc_bwd_nc_a_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_g,
                   const __grid_constant__ CUtensorMap map_dq, const NcBwdParams prm) {
  using G = NA<D>;
  constexpr int ST = G::ST;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sbuf = sm + G::OFF_SBUF;
  float* zn = reinterpret_cast<float*>(sm + G::OFF_ZN);
  float* vn = reinterpret_cast<float*>(sm + G::OFF_VN);
  float* barr = reinterpret_cast<float*>(sm + G::OFF_BARR);
  float* carr = reinterpret_cast<float*>(sm + G::OFF_CARR);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + G::OFF_BAR);
  uint64_t* full = bars;               // [ST]
  uint64_t* phi_done = bars + ST;      // [ST]
  uint64_t* empty = bars + 2 * ST;     // [ST] MMAs of the stage's chunk done
  uint64_t* ost_full = bars + 3 * ST;  // [ST] dq staged (group D)
  uint64_t* rdone = bars + 4 * ST;     // [ST] r sums read the stage (group A)
  uint64_t* b_ready = bars + 5 * ST;   // [ST] b of the stage's chunk written (group B)
  uint64_t* x = bars + 6 * ST;
  uint64_t* o_full = x;                // [2]
  uint64_t* a_ready = x + 2;           // [2]
  uint64_t* dq_full = x + 4;           // [2]
  uint64_t* dq_empty = x + 6;          // [2]
  uint64_t* s_ready = x + 8;
  uint64_t* mma_fin = x + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + G::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + G::OFF_MISC + 4);
  // pass B may start filling its pipeline while this grid runs
  griddep_launch_dependents();
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(prm.status);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / prm.P, seg = blockIdx.x % prm.P;
  const int tok0 = seg * prm.seg_len;
  const int tok_end = min(prm.N, tok0 + prm.seg_len);
  const int nchunks = (tok_end - tok0 + C - 1) / C;
  const long long rstride = rec_words<D>();
  const float* recs = prm.ws_state + (long long)bh * prm.P * prm.F * rstride;
  const int nrec = prm.P * prm.F;
  float* rec_out = prm.ws_rev + ((long long)bh * prm.P + seg) * rstride;

  if (tid == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&phi_done[i], 128);
      mbar_init(&empty[i], 1);
      mbar_init(&ost_full[i], 128);
      mbar_init(&rdone[i], 128);
      mbar_init(&b_ready[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&a_ready[i], 128);
      mbar_init(&dq_full[i], 1);
      mbar_init(&dq_empty[i], 128);
    }
    mbar_init(s_ready, 128);
    mbar_init(mma_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_g);
      tma_prefetch_desc(&map_dq);
      // the stage of chunk c is free once its MMAs, its dq epilogue and its
      // r sums are done; its dq (in the dead G tile) is stored first
      auto retire = [&](int c) -> bool {
        const int s = c % ST;
        const uint32_t par = (c / ST) & 1;
        if (!mbar_wait(&empty[s], par, abort_flag, kTimeoutNs) ||
            !mbar_wait(&ost_full[s], par, abort_flag, kTimeoutNs) ||
            !mbar_wait(&rdone[s], par, abort_flag, kTimeoutNs))
          return false;
        tma_store_3d(&map_dq, sm + s * G::STAGE + G::OFF_G, 0, tok0 + c * C, bh);
        tma_store_commit();
        tma_store_wait_read<0>();
        return true;
      };
      int issued = 0;
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST;
        if (c >= ST && !(ok = retire(c - ST))) break;
        uint8_t* stg = sm + s * G::STAGE;
        mbar_arrive_expect_tx(&full[s], 2 * G::TILE);
        tma_load_3d(stg, &map_q, &full[s], 0, tok0 + c * C, bh);
        tma_load_3d(stg + G::OFF_G, &map_g, &full[s], 0, tok0 + c * C, bh);
        issued = c + 1;
      }
      for (int c = max(0, issued - ST); c < issued && ok; ++c) ok = retire(c);
      tma_store_wait<0>();
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_drain(&full[c % ST], (c / ST) & 1, kTimeoutNs);
    }
  } else if (warp == 13) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_qs = make_idesc_bf16(128, G::NO, false, false);  // [O | den] = phiQ [S_N^T ; z]^T
      constexpr uint32_t id_as = make_idesc_bf16(128, D, false, true);       // dQ = a S_N^T (copy MN-major)
      constexpr uint32_t id_tt = make_idesc_bf16(D, D, true, true);          // R += phiQ^T a
      const uint32_t sb = smem_u32(sbuf);
      const uint64_t dsk = make_sdesc(sb, 16, 1024, kSwizzle128B);
      const uint64_t dsm = make_sdesc(sb, D * 128, 1024, kSwizzle128B);
      // [O | den] of chunk c + 1 is issued before the wait for chunk c's row
      // pass, so that the row pass of c + 1 can follow that of c at once; its
      // buffer was last read by the row pass of c - 1, which the issuer has
      // already waited for
      auto issue_o = [&](int c) -> bool {
        const int s = c % ST, ob = c & 1;
        if (!mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs)) return false;
        tc_fence_after();
        const uint64_t dq = make_sdesc(smem_u32(sm + s * G::STAGE), 16, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + G::col_o(ob), sdesc_add(dq, k * 32), sdesc_add(dsk, k * 32), id_qs, k > 0);
        tc_commit(&o_full[ob]);
        return true;
      };
      bool ok = mbar_wait(s_ready, 0, abort_flag, kTimeoutNs);
      if (ok && nchunks > 0) ok = issue_o(0);
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST, ob = c & 1;
        const uint32_t qa = smem_u32(sm + s * G::STAGE), ga = qa + G::OFF_G;
        if (c + 1 < nchunks && !(ok = issue_o(c + 1))) break;
        ok = mbar_wait(&a_ready[ob], (c >> 1) & 1, abort_flag, kTimeoutNs);
        if (ok && c >= 2) ok = mbar_wait(&dq_empty[ob], ((c >> 1) - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dg = make_sdesc(ga, 16, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + G::col_dq(ob), sdesc_add(dg, k * 32), sdesc_add(dsm, k * 2048), id_as, k > 0);
        const uint64_t dqm = make_sdesc(qa, BOX, 1024, kSwizzle128B);
        const uint64_t dgm = make_sdesc(ga, BOX, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ss(tmem + G::COL_R, sdesc_add(dqm, k * 2048), sdesc_add(dgm, k * 2048), id_tt,
                 (c > 0 || k > 0) ? 1u : 0u);
        // dq_full covers the R MMA too: the epilogue overwrites a
        tc_commit(&dq_full[ob]);
        tc_commit(&empty[s]);
      }
      tc_commit(mma_fin);
      mbar_drain(mma_fin, 0, kTimeoutNs);
    }
  } else if (warp < 4) {
    // ---------------- group A: phi(Q), totals, r, R ----------------
    using X = ExactLayout<D, 128>;
    const int t = tid;
    const int q = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    const int fc = X::FCW * (t >> 5) + (lane % X::FCW);
    float racc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) racc[e] = 0.f;
    griddep_wait();
    sum_states_to_tmem<D>(recs, rstride, 0, nrec, lane_addr, G::COL_S, row);
    copy_state_to_smem<D>(lane_addr + G::COL_S, sbuf, row);
    // z_psi,N: fp32 for the epilogue; as bf16 hi + lo rows D, D + 1 of the MMA
    // operand (phi(q).z_psi = phi(q).z_hi + phi(q).z_lo, about 16 bits); row
    // D + 2 ones (s_t); rows D + 3 .. zero. The sum of all v for the row pass.
    if (t < D) {
      const float acc = sum_vector_entry<D>(recs, rstride, 0, nrec, t);
      zn[t] = acc;
      vn[t] = sum_vector_entry<D>(recs, rstride, 0, nrec, D + t);
      const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
      const __nv_bfloat16 lo = __float2bfloat16_rn(acc - __bfloat162float(hi));
      *reinterpret_cast<__nv_bfloat16*>(sbuf + sw128(D, t >> 3) + 2 * (t & 7)) = hi;
      *reinterpret_cast<__nv_bfloat16*>(sbuf + sw128(D + 1, t >> 3) + 2 * (t & 7)) = lo;
      *reinterpret_cast<__nv_bfloat16*>(sbuf + sw128(D + 2, t >> 3) + 2 * (t & 7)) = __float2bfloat16_rn(1.f);
    }
    for (int i = t; i < (G::NO - D - 3) * 8; i += 128)
      *reinterpret_cast<uint4*>(sbuf + sw128(D + 3 + (i >> 3), i & 7)) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(s_ready);
    bool ok = true;
    for (int c = 0; c <= nchunks && ok; ++c) {
      if (c < nchunks) {
        const int s = c % ST;
        ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        phi_tile_bf16<D, 128>(sm + s * G::STAGE, t);
        fence_proxy_async_smem();
        mbar_arrive(&phi_done[s]);
      }
      if (c >= 1) {
        // r += sum_t b_t phi(q_t) over the previous chunk
        const int cp = c - 1, sp = cp % ST;
        ok = mbar_wait(&a_ready[cp & 1], (cp >> 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        wcolsum_tile<D, 128>(sm + sp * G::STAGE, barr + sp * C, t, racc);
        mbar_arrive(&rdone[sp]);
      }
    }
    reduce_row_groups<D, 128>(racc);
    if (ok && lane < X::FCW) {
      float4* rd = reinterpret_cast<float4*>(rec_out + D * D + 8 * fc);
      rd[0] = make_float4(racc[0], racc[1], racc[2], racc[3]);
      rd[1] = make_float4(racc[4], racc[5], racc[6], racc[7]);
    }
    if (ok) ok = mbar_wait(mma_fin, 0, abort_flag, kTimeoutNs);
    if (ok) {
      tc_fence_after();
      store_state_from_tmem<D>(rec_out, lane_addr, G::COL_R, row);
    }
  } else if (warp < 8) {
    // ---------------- group B: a and b from [O | den] ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST, ob = c & 1;
      uint8_t* stg = sm + s * G::STAGE;
      ok = mbar_wait(&o_full[ob], (c >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      uint32_t dz[2], sq;
      tmem_ld2(lane_addr + G::col_o(ob) + D, dz);
      tmem_ld1(lane_addr + G::col_o(ob) + D + 2, sq);
      tmem_ld_wait();
      const float srow = __uint_as_float(sq);
      const float nt = (float)prm.N;
      const float den = fmaf(srow, nt, __uint_as_float(dz[0]) + __uint_as_float(dz[1])) + prm.eps;
      const float inv_den = 1.f / den;
      float beta0;
      const float beta1 = grad_row_pass_centred<D>(lane_addr + G::col_o(ob), stg + G::OFF_G, r, inv_den, vn, &beta0);
      const float b = -fmaf(srow, beta0, beta1) / den;
      barr[s * C + r] = b;
      carr[s * C + r] = fmaf(nt, b, beta0);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&a_ready[ob]);
      mbar_arrive(&b_ready[s]);
    }
  } else {
    // ---------------- group D: dq ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    bool ok = mbar_wait(s_ready, 0, abort_flag, kTimeoutNs);     // zn
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST, ob = c & 1;
      uint8_t* stg = sm + s * G::STAGE;
      // b of the chunk from group B (per stage: group B cannot refill the
      // stage before this epilogue is done); then dQ (and the R update,
      // which reads a) done
      ok = mbar_wait(&b_ready[s], (c / ST) & 1, abort_flag, kTimeoutNs) &&
           mbar_wait(&dq_full[ob], (c >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      // dq staged in the dead G tile; the producer stores it before
      // refilling the stage
      grad_epilogue<D>(lane_addr + G::col_dq(ob), stg, r, barr[s * C + r], zn, stg + G::OFF_G, carr[s * C + r]);
      tc_fence_before();
      mbar_arrive(&dq_empty[ob]);
      fence_proxy_async_smem();
      mbar_arrive(&ost_full[s]);
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  // after the barrier: a warp that gave up late is seen too
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

template <int D>
struct NB {
  static_assert(D == 64, "the tensor-core backward is laid out for D = 64");
  static constexpr int TILE = BOX;
  static constexpr int ST = 4;                        // stages of K, V
  static constexpr int OFF_V = TILE;
  static constexpr int STAGE = 2 * TILE;
  static constexpr int OFF_RBUF = ST * STAGE;         // bf16 R_0 copy, D rows
  static constexpr int OFF_RVEC = OFF_RBUF + D * 128; // [D] r_0
  static constexpr int OFF_BAR = OFF_RVEC + D * 4;
  static constexpr int NBAR = 4 * ST + 4 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
  static constexpr uint32_t COL_R = 0;                // R_0 (M = D layout)
  __host__ __device__ static constexpr uint32_t col_dk(int ob) { return D + 2 * D * ob; }
  __host__ __device__ static constexpr uint32_t col_dv(int ob) { return 2 * D + 2 * D * ob; }
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(col_dv(1) + D <= TMEM_COLS, "tensor memory budget");
};

struct NcBwdBParams {
  int N, P, seg_len;
  const float* ws_rev;     // [BH][P][rec_words] (R, r) of every segment
  int* status;
};

// Pass B. Warps 0-3: phi(K) in place; warps 4-7: the R_0 / r_0 sums and the
// R_0 copy, then the dk, dv epilogue (dk staged in the dead V tile, dv in the
// dead K tile, row by row); warp 8 TMA; warp 9 TMEM and MMA.
template <int D>
__global__ void __launch_bounds__(320, 1)
tc_bwd_nc_b_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
                   const NcBwdBParams prm) {
  using G = NB<D>;
  constexpr int ST = G::ST;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* rbuf = sm + G::OFF_RBUF;
  float* rvec = reinterpret_cast<float*>(sm + G::OFF_RVEC);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + G::OFF_BAR);
  uint64_t* full = bars;               // [ST]
  uint64_t* phi_done = bars + ST;      // [ST]
  uint64_t* empty = bars + 2 * ST;     // [ST] MMAs of the stage's chunk done
  uint64_t* ost_full = bars + 3 * ST;  // [ST] dk, dv staged
  uint64_t* x = bars + 4 * ST;
  uint64_t* kv_full = x;               // [2]
  uint64_t* kv_empty = x + 2;          // [2]
  uint64_t* r_ready = x + 4;
  uint64_t* mma_fin = x + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + G::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + G::OFF_MISC + 4);
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(prm.status);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / prm.P, seg = blockIdx.x % prm.P;
  const int tok0 = seg * prm.seg_len;
  const int tok_end = min(prm.N, tok0 + prm.seg_len);
  const int nchunks = (tok_end - tok0 + C - 1) / C;
  const long long rstride = rec_words<D>();
  const float* recs = prm.ws_rev + (long long)bh * prm.P * rstride;

  if (tid == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&phi_done[i], 128);
      mbar_init(&empty[i], 1);
      mbar_init(&ost_full[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 128);
    }
    mbar_init(r_ready, 128);
    mbar_init(mma_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      tma_prefetch_desc(&map_dk);
      tma_prefetch_desc(&map_dv);
      auto retire = [&](int c) -> bool {
        const int s = c % ST;
        const uint32_t par = (c / ST) & 1;
        if (!mbar_wait(&empty[s], par, abort_flag, kTimeoutNs) ||
            !mbar_wait(&ost_full[s], par, abort_flag, kTimeoutNs))
          return false;
        uint8_t* stg = sm + s * G::STAGE;
        tma_store_3d(&map_dk, stg + G::OFF_V, 0, tok0 + c * C, bh);
        tma_store_3d(&map_dv, stg, 0, tok0 + c * C, bh);
        tma_store_commit();
        tma_store_wait_read<0>();
        return true;
      };
      int issued = 0;
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST;
        if (c >= ST && !(ok = retire(c - ST))) break;
        uint8_t* stg = sm + s * G::STAGE;
        mbar_arrive_expect_tx(&full[s], 2 * G::TILE);
        tma_load_3d(stg, &map_k, &full[s], 0, tok0 + c * C, bh);
        tma_load_3d(stg + G::OFF_V, &map_v, &full[s], 0, tok0 + c * C, bh);
        issued = c + 1;
      }
      for (int c = max(0, issued - ST); c < issued && ok; ++c) ok = retire(c);
      tma_store_wait<0>();
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_drain(&full[c % ST], (c / ST) & 1, kTimeoutNs);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_vr = make_idesc_bf16(128, D, false, false);   // dK = V R_0^T (R copy K-major)
      constexpr uint32_t id_kr = make_idesc_bf16(128, D, false, true);    // dV = phiK R_0 (copy MN-major)
      const uint32_t rb = smem_u32(rbuf);
      const uint64_t drk = make_sdesc(rb, 16, 1024, kSwizzle128B);
      const uint64_t drm = make_sdesc(rb, D * 128, 1024, kSwizzle128B);
      bool ok = mbar_wait(r_ready, 0, abort_flag, kTimeoutNs);
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST, ob = c & 1;
        const uint32_t ka = smem_u32(sm + s * G::STAGE), va = ka + G::OFF_V;
        ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (ok && c >= 2) ok = mbar_wait(&kv_empty[ob], ((c >> 1) - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dv_ = make_sdesc(va, 16, 1024, kSwizzle128B);
        const uint64_t dk_ = make_sdesc(ka, 16, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + G::col_dk(ob), sdesc_add(dv_, k * 32), sdesc_add(drk, k * 32), id_vr, k > 0);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + G::col_dv(ob), sdesc_add(dk_, k * 32), sdesc_add(drm, k * 2048), id_kr, k > 0);
        tc_commit(&kv_full[ob]);
        tc_commit(&empty[s]);
      }
      tc_commit(mma_fin);
      mbar_drain(mma_fin, 0, kTimeoutNs);
    }
  } else if (warp < 4) {
    // ---------------- group C: phi(K) ----------------
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      phi_tile_bf16<D, 128>(sm + s * G::STAGE, tid);
      fence_proxy_async_smem();
      mbar_arrive(&phi_done[s]);
    }
  } else {
    // ---------------- group E: R_0, r_0; dk, dv ----------------
    const int t = tid - 128;
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    griddep_wait();
    sum_states_to_tmem<D>(recs, rstride, 0, prm.P, lane_addr, G::COL_R, row);
    tc_fence_before();
    tc_fence_after();
    copy_state_to_smem<D>(lane_addr + G::COL_R, rbuf, row);
    for (int i = t; i < D; i += 128) {
      float acc = 0.f;
      for (int p = 0; p < prm.P; ++p) acc += recs[p * rstride + D * D + i];
      rvec[i] = acc;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(r_ready);
    bool ok = mbar_wait(r_ready, 0, abort_flag, kTimeoutNs);   // rvec complete
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST, ob = c & 1;
      uint8_t* stg = sm + s * G::STAGE;
      ok = mbar_wait(&kv_full[ob], (c >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      // dk = (dK + r_0) phi'(k) into the V tile, then dv into this row of
      // the K tile (the row's phi(k) has been read)
      grad_epilogue<D>(lane_addr + G::col_dk(ob), stg, r, 1.f, rvec, stg + G::OFF_V);
      store_row_bf16<D>(lane_addr + G::col_dv(ob), stg, r);
      tc_fence_before();
      mbar_arrive(&kv_empty[ob]);
      fence_proxy_async_smem();
      mbar_arrive(&ost_full[s]);
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  // after the barrier: a warp that gave up late is seen too
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <typename Kernel, typename... Args>
cudaError_t launch_dependent(Kernel kernel, int grid, int threads, int smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

template <int D>
cudaError_t launch_backward(const BwdArgs& a) {
  FwdArgs f{};
  f.q = a.q; f.k = a.k; f.v = a.v; f.out = nullptr;
  f.BH = a.BH; f.N = a.N; f.dk = a.dk; f.dv = a.dv; f.causal = a.causal;
  f.eps = a.eps; f.dtype = a.dtype; f.ws_state = a.ws_state; f.plan = a.plan;
  f.stream = a.stream;
  cudaError_t e = cudaSuccess;
  if (!a.state_ready) {
    prof_begin(LA_SPAN_BWD_STATE, a.stream);
    e = tc_segment_state(f);              // sums of S^T, z for segments 0 .. P-2
    prof_end(LA_SPAN_BWD_STATE, a.stream);
    if (e != cudaSuccess) return e;
  }

  CUtensorMap mq, mk, mv, mg;
  e = make_map(&mq, a.q, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mk, a.k, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mv, a.v, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mg, a.dout, a.BH, a.N, D);
  CUtensorMap mdq, mdk, mdv;
  if (e == cudaSuccess) e = make_map(&mdq, a.dq, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mdk, a.dk_, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mdv, a.dv_, a.BH, a.N, D);
  if (e != cudaSuccess) return e;
  int* status = device_status_ptr();

  constexpr int smem1 = B1<D>::BYTES;
  e = cudaFuncSetAttribute(tc_bwd1_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem1);
  if (e != cudaSuccess) return e;
  Bwd1Params p1{a.N, a.plan.P, a.plan.seg_len, a.plan.F, a.eps, a.ws_state, a.ws_rev, a.ws_tok, (__nv_bfloat16*)a.dq, status};
  prof_begin(LA_SPAN_BWD_SWEEP1, a.stream);
  e = launch_dependent(tc_bwd1_kernel<D>, a.BH * a.plan.P, B1<D>::THREADS, smem1, a.stream, mq, mk, mv, mg, mdq, p1);
  prof_end(LA_SPAN_BWD_SWEEP1, a.stream);
  if (e != cudaSuccess) return e;
  note_launch();

  constexpr int smem2 = B2<D>::BYTES;
  e = cudaFuncSetAttribute(tc_bwd2_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2);
  if (e != cudaSuccess) return e;
  Bwd2Params p2{a.N, a.plan.P, a.plan.seg_len, a.ws_rev, a.ws_tok, (__nv_bfloat16*)a.dk_, (__nv_bfloat16*)a.dv_,
                status};
  prof_begin(LA_SPAN_BWD_SWEEP2, a.stream);
  e = launch_dependent(tc_bwd2_kernel<D>, a.BH * a.plan.P, B2<D>::THREADS, smem2, a.stream, mq, mk, mv, mg, mdk, mdv,
                       p2);
  prof_end(LA_SPAN_BWD_SWEEP2, a.stream);
  if (e == cudaSuccess) note_launch();
  return e;
}

// Non-causal: the state pass over every segment (S_N, z_N records), then
// pass A (dq, (R, r) records) and pass B (dk, dv), each a dependent of the
// launch before it.
template <int D>
cudaError_t launch_backward_nc(const BwdArgs& a) {
  FwdArgs f{};
  f.q = a.q; f.k = a.k; f.v = a.v; f.out = nullptr;
  f.BH = a.BH; f.N = a.N; f.dk = a.dk; f.dv = a.dv; f.causal = 0;
  f.eps = a.eps; f.dtype = a.dtype; f.ws_state = a.ws_state; f.plan = a.plan;
  f.stream = a.stream;
  cudaError_t e = cudaSuccess;
  if (!a.state_ready) {
    prof_begin(LA_SPAN_BWD_STATE, a.stream);
    e = tc_segment_state(f);              // sums of S^T, z for every segment
    prof_end(LA_SPAN_BWD_STATE, a.stream);
    if (e != cudaSuccess) return e;
  }

  CUtensorMap mq, mk, mv, mg, mdq, mdk, mdv;
  e = make_map(&mq, a.q, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mk, a.k, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mv, a.v, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mg, a.dout, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mdq, a.dq, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mdk, a.dk_, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mdv, a.dv_, a.BH, a.N, D);
  if (e != cudaSuccess) return e;
  int* status = device_status_ptr();

  constexpr int smema = NA<D>::BYTES;
  e = cudaFuncSetAttribute(tc_bwd_nc_a_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smema);
  if (e != cudaSuccess) return e;
  NcBwdParams pa{a.N, a.plan.P, a.plan.seg_len, a.plan.F, a.eps, a.ws_state, a.ws_rev, status};
  prof_begin(LA_SPAN_BWD_SWEEP1, a.stream);
  e = launch_dependent(tc_bwd_nc_a_kernel<D>, a.BH * a.plan.P, NA<D>::THREADS, smema, a.stream, mq, mg, mdq, pa);
  prof_end(LA_SPAN_BWD_SWEEP1, a.stream);
  if (e != cudaSuccess) return e;
  note_launch();

  constexpr int smemb = NB<D>::BYTES;
  e = cudaFuncSetAttribute(tc_bwd_nc_b_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smemb);
  if (e != cudaSuccess) return e;
  NcBwdBParams pb{a.N, a.plan.P, a.plan.seg_len, a.ws_rev, status};
  prof_begin(LA_SPAN_BWD_SWEEP2, a.stream);
  e = launch_dependent(tc_bwd_nc_b_kernel<D>, a.BH * a.plan.P, 320, smemb, a.stream, mk, mv, mdk, mdv, pb);
  prof_end(LA_SPAN_BWD_SWEEP2, a.stream);
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace

bool tc_backward_supported(int dk, int dv, la_dtype dtype, int causal) {
  (void)causal;
  return dtype == LA_BF16 && dk == 64 && dv == 64;
}

cudaError_t tc_backward(const BwdArgs& a) { return a.causal ? launch_backward<64>(a) : launch_backward_nc<64>(a); }

}  // namespace la
