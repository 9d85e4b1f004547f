// Pieces shared by the tensor-core kernels (forward and backward): chunk and
// box geometry, the 128-byte swizzle, phi on operand tiles in shared memory,
// state copies from tensor memory, and the TMA tensor maps of [BH][N][D] bf16
// inputs. Included by one translation unit per kernel family; everything has
// internal linkage.
#pragma once

#include <cudaTypedefs.h>

#include "la_internal.cuh"
#include "la_sm100.cuh"

namespace la {
namespace {

using namespace sm100;

constexpr int C = 128;                    // tokens per chunk
constexpr int BOX = 128 * 128;            // bytes of one [128 rows][64 bf16] SW128 box
constexpr uint64_t kTimeoutNs = 2000000000ull;

// Floats per state record of the tensor-core kernels: [D x D | D | D]. At
// D = 64 (causal and non-causal, no decay) the state pass writes centred sums
// over its tokens: S_psi^T = V^T psi(K) and z_psi = sum psi(k) with
// psi = phi - 1, then the plain sum of the values v; the full state is
// S^T = S_psi^T + (sum v) 1^T, z = z_psi + n 1 (n the number of tokens). The
// large common part of phi(k) (its 1) is thus carried exactly in fp32, and
// only the small part psi goes through bf16 operands. Otherwise the record is
// [S^T | z | unused].
template <int D>
__host__ __device__ constexpr long long rec_words() { return (long long)D * D + 2 * D; }

// Row of the D x D state held by lane `l` of TMEM quadrant `q` (rows live in
// the quadrant's lanes: all 32 for M = 128, the first 16 for M = 64).
template <int D>
__device__ __forceinline__ int state_row(int q, int l) {
  if (D == 128) return 32 * q + l;
  return l < 16 ? 16 * q + l : -1;
}

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {  // byte offset of a 16-byte chunk
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void report_timeout(int* status) { atomicExch(status, (int)LA_ERR_TIMEOUT); }

// phi on packed bf16 values, in place on one [C][D] tile (phi is elementwise,
// so the swizzle does not matter); NT threads, thread t owns 16-byte chunks
// t, t + NT, ...
template <int D, int NT>
__device__ __forceinline__ void phi_tile_bf16(uint8_t* tile, int t) {
  constexpr int PER = (C * D * 2 / 16) / NT;
  constexpr int GR = 4;
#pragma unroll 1
  for (int i0 = 0; i0 < PER; i0 += GR) {
    uint4 w[GR];
#pragma unroll
    for (int i = 0; i < GR; ++i) w[i] = reinterpret_cast<const uint4*>(tile)[t + NT * (i0 + i)];
#pragma unroll
    for (int i = 0; i < GR; ++i) {
      w[i].x = phi_bf16x2(w[i].x);
      w[i].y = phi_bf16x2(w[i].y);
      w[i].z = phi_bf16x2(w[i].z);
      w[i].w = phi_bf16x2(w[i].w);
    }
#pragma unroll
    for (int i = 0; i < GR; ++i) reinterpret_cast<uint4*>(tile)[t + NT * (i0 + i)] = w[i];
  }
}

// phi(x) in fp32 without branches: x + 1 for x > 0, e^x otherwise, with
// e^x = 2^(x log2 e) from the hardware base-2 exponential. Values below
// 2^-62 are raised to 2^-62 (as in phi_bf16x2): phi stays positive and the
// product of two features a normal fp32 number. Rounded to bf16 by the
// caller.
__device__ __forceinline__ float phi_f32(float x) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * 1.4426950408889634f));
  return x > 0.f ? x + 1.f : fmaxf(e, 2.16840434e-19f);
}

// psi(x) = phi(x) - 1: x for x > 0 (exact), e^x - 1 otherwise (the
// subtraction is exact in fp32 for e^x in [1/2, 1]; below that the absolute
// error stays at the exponential's own, ~2^-22).
__device__ __forceinline__ float psi_f32(float x) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * 1.4426950408889634f));
  return x > 0.f ? x : e - 1.f;
}

// phi in place on one [C][D] tile, rounded to nearest, with fp32 column sums
// over rows < n_valid (rows >= n_valid, past the end of the sequence, become
// zero). NT threads; warp w owns FCW = D / (NT / 4) consecutive 16-byte
// feature chunks of every row; lane l works on chunk FCW*w + l % FCW and rows
// l / FCW + (32 / FCW) i. The column sums are reduced inside the warp, so on
// return lanes l < FCW hold the sums of the 8 features of chunk FCW*w + l.
template <int D, int NT>
struct ExactLayout {
  static constexpr int FCW = D / (NT / 4);     // feature chunks per warp
  static constexpr int RG = 32 / FCW;          // row groups per warp
  static constexpr int RPT = C / RG;           // rows per thread
  static_assert(FCW >= 1 && FCW <= 8 && (FCW & (FCW - 1)) == 0, "layout");
};

template <int D, int NT, bool kCheck, bool kSum, bool kScale = false, bool kPsi = false>
__device__ __forceinline__ void phi_tile_exact_rows(uint8_t* base, int ch, int r0, int n_valid, float (&zacc)[8],
                                                    float log2a = 0.f, int wbase = 0) {
  using X = ExactLayout<D, NT>;
  constexpr int GR = 4;                               // rows per loop trip (kept small: code size)
#pragma unroll 1
  for (int i0 = 0; i0 < X::RPT; i0 += GR) {
    uint4 wv[GR];
#pragma unroll
    for (int i = 0; i < GR; ++i) wv[i] = *reinterpret_cast<const uint4*>(base + sw128(r0 + X::RG * (i0 + i), ch));
#pragma unroll
    for (int i = 0; i < GR; ++i) {
      const int rr = r0 + X::RG * (i0 + i);
      const bool valid = !kCheck || rr < n_valid;
      // kScale: row rr is weighted by 2^((wbase - rr) log2a) = a^(wbase - rr)
      const float w = kScale ? (valid ? exp2f((float)(wbase - rr) * log2a) : 0.f) : 1.f;
      uint32_t* p = reinterpret_cast<uint32_t*>(&wv[i]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float lo = valid ? (kPsi ? psi_f32(__uint_as_float(p[h] << 16)) : phi_f32(__uint_as_float(p[h] << 16))) : 0.f;
        float hi = valid ? (kPsi ? psi_f32(__uint_as_float(p[h] & 0xFFFF0000u))
                                 : phi_f32(__uint_as_float(p[h] & 0xFFFF0000u)))
                         : 0.f;
        if (kScale) {
          lo *= w;
          hi *= w;
        }
        if (kSum) {
          zacc[2 * h] += lo;
          zacc[2 * h + 1] += hi;
        }
        p[h] = pack_bf16x2(lo, hi);
      }
    }
#pragma unroll
    for (int i = 0; i < GR; ++i) *reinterpret_cast<uint4*>(base + sw128(r0 + X::RG * (i0 + i), ch)) = wv[i];
  }
}

// kReduce: zacc is cleared first and, on return, reduced inside the warp as
// above. Otherwise this thread's partial sums are added to zacc, and the
// caller reduces them (reduce_row_groups) when it needs the totals.
// kSum = false: phi only, zacc untouched. kScale: row r (of the tile) is
// multiplied by a^(wbase - r), a = 2^log2a (decay weights), before rounding.
// kPsi: psi = phi - 1 instead of phi (and its column sums).
template <int D, int NT, bool kReduce = true, bool kSum = true, bool kScale = false, bool kPsi = false>
__device__ __forceinline__ void phi_tile_exact(uint8_t* tile, int t, int n_valid, float (&zacc)[8],
                                               float log2a = 0.f, int wbase = 0) {
  using X = ExactLayout<D, NT>;
  const int w = t >> 5, lane = t & 31;
  const int fc = X::FCW * w + (lane % X::FCW);       // feature chunk 0 .. D/8-1
  const int r0 = lane / X::FCW;
  uint8_t* base = tile + (fc >> 3) * BOX;
  const int ch = fc & 7;
  if (kReduce && kSum) {
#pragma unroll
    for (int e = 0; e < 8; ++e) zacc[e] = 0.f;
  }
  // full tiles skip the per-row validity test
  if (n_valid >= C)
    phi_tile_exact_rows<D, NT, false, kSum, kScale, kPsi>(base, ch, r0, n_valid, zacc, log2a, wbase);
  else
    phi_tile_exact_rows<D, NT, true, kSum, kScale, kPsi>(base, ch, r0, n_valid, zacc, log2a, wbase);
  if (kReduce && kSum) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float x = zacc[e];
#pragma unroll
      for (int o = X::FCW; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      zacc[e] = x;
    }
  }
}

// Weighted column sums over one [C][D] bf16 tile in the ExactLayout mapping:
// acc[e] += sum over this thread's rows r of w[r] * tile[r][8 fc + e]. The
// sums are per thread; reduce_row_groups finishes them inside the warp.
template <int D, int NT>
__device__ __forceinline__ void wcolsum_tile(const uint8_t* tile, const float* w, int t, float (&acc)[8]) {
  using X = ExactLayout<D, NT>;
  constexpr int GR = 4;
  const int wi = t >> 5, lane = t & 31;
  const int fc = X::FCW * wi + (lane % X::FCW);
  const int r0 = lane / X::FCW;
  const uint8_t* base = tile + (fc >> 3) * BOX;
  const int ch = fc & 7;
#pragma unroll 1
  for (int i0 = 0; i0 < X::RPT; i0 += GR) {
    uint4 wv[GR];
    float wr[GR];
#pragma unroll
    for (int i = 0; i < GR; ++i) {
      const int r = r0 + X::RG * (i0 + i);
      wv[i] = *reinterpret_cast<const uint4*>(base + sw128(r, ch));
      wr[i] = w[r];
    }
#pragma unroll
    for (int i = 0; i < GR; ++i) {
      const uint32_t* p = reinterpret_cast<const uint32_t*>(&wv[i]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        acc[2 * h] = fmaf(wr[i], __uint_as_float(p[h] << 16), acc[2 * h]);
        acc[2 * h + 1] = fmaf(wr[i], __uint_as_float(p[h] & 0xFFFF0000u), acc[2 * h + 1]);
      }
    }
  }
}

// Plain column sums over one [C][D] bf16 tile in the ExactLayout mapping:
// acc[e] += sum over this thread's rows r < n_valid of tile[r][8 fc + e].
template <int D, int NT>
__device__ __forceinline__ void colsum_tile(const uint8_t* tile, int t, int n_valid, float (&acc)[8]) {
  using X = ExactLayout<D, NT>;
  constexpr int GR = 4;
  const int wi = t >> 5, lane = t & 31;
  const int fc = X::FCW * wi + (lane % X::FCW);
  const int r0 = lane / X::FCW;
  const uint8_t* base = tile + (fc >> 3) * BOX;
  const int ch = fc & 7;
#pragma unroll 1
  for (int i0 = 0; i0 < X::RPT; i0 += GR) {
    uint4 wv[GR];
#pragma unroll
    for (int i = 0; i < GR; ++i) {
      const int r = r0 + X::RG * (i0 + i);
      wv[i] = r < n_valid ? *reinterpret_cast<const uint4*>(base + sw128(r, ch)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < GR; ++i) {
      const uint32_t* p = reinterpret_cast<const uint32_t*>(&wv[i]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        acc[2 * h] += __uint_as_float(p[h] << 16);
        acc[2 * h + 1] += __uint_as_float(p[h] & 0xFFFF0000u);
      }
    }
  }
}

// Sum the per-thread column sums of the ExactLayout mapping over the row
// groups of the warp; lanes l < FCW end with the totals of chunk FCW*w + l.
template <int D, int NT>
__device__ __forceinline__ void reduce_row_groups(float (&acc)[8]) {
  using X = ExactLayout<D, NT>;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float x = acc[e];
#pragma unroll
    for (int o = X::FCW; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    acc[e] = x;
  }
}

// Copy this thread's TMEM lane of a D x D state (fp32, D columns starting at
// tensor-memory address `taddr`) to a bf16 operand buffer laid out as boxes of
// [D rows][64 columns] with 128-byte swizzle (row = first index of the state).
// Read as MN-major it is the state with the column index along N; read as
// K-major it is the state with the row index along N.
template <int D>
__device__ __forceinline__ void copy_state_to_smem(uint32_t taddr, uint8_t* sbuf, int row) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(taddr + c0, v);
    tmem_ld_wait();
    if (row >= 0) {
      const int b = c0 / 64, cb = (c0 % 64) / 8;  // box, first 16-byte chunk
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
        w.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
        w.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
        w.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
        *reinterpret_cast<uint4*>(sbuf + b * (D * 128) + sw128(row, cb + j)) = w;
      }
    }
  }
}

// A D x D fp32 state from global memory (row-major) into tensor memory at
// column `col` (rows in the M = D accumulator layout).
template <int D>
__device__ __forceinline__ void load_state_to_tmem(const float* src, uint32_t lane_addr, uint32_t col, int row) {
  const float4* srow = reinterpret_cast<const float4*>(src + (row >= 0 ? row : 0) * D);
#pragma unroll
  for (int h = 0; h < D; h += 64) {
    float4 f[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = row >= 0 ? srow[h / 4 + j] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[4 * j + 0] = __float_as_uint(f[4 * g + j].x);
        v[4 * j + 1] = __float_as_uint(f[4 * g + j].y);
        v[4 * j + 2] = __float_as_uint(f[4 * g + j].z);
        v[4 * j + 3] = __float_as_uint(f[4 * g + j].w);
      }
      tmem_st16(lane_addr + col + h + 16 * g, v);
    }
  }
  tmem_st_wait();
}

// A D x D fp32 state from tensor memory (column `col`) to global memory.
template <int D>
__device__ __forceinline__ void store_state_from_tmem(float* dst, uint32_t lane_addr, uint32_t col, int row) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(lane_addr + col + c0, v);
    tmem_ld_wait();
    if (row >= 0) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(dst + row * D + c0 + j) =
            make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                        __uint_as_float(v[j + 3]));
    }
  }
}

// Sum of the D x D parts of the state records p0 .. p1-1 (`stride` floats
// apart, row-major) for this thread's state row, plus `add` in every entry,
// into tensor memory at column `col` (rows in the M = D accumulator layout;
// row < 0: lane unused).
template <int D>
__device__ __forceinline__ void sum_states_to_tmem(const float* recs, long long stride, int p0, int p1,
                                                   uint32_t lane_addr, uint32_t col, int row, float add = 0.f) {
#pragma unroll 1
  for (int h = 0; h < D; h += 64) {
    float4 acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = make_float4(add, add, add, add);
    if (row >= 0) {
#pragma unroll 1
      for (int p = p0; p < p1; ++p) {
        const float4* src = reinterpret_cast<const float4*>(recs + p * stride + (long long)row * D + h);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float4 f = src[j];
          acc[j].x += f.x; acc[j].y += f.y; acc[j].z += f.z; acc[j].w += f.w;
        }
      }
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[4 * j + 0] = __float_as_uint(acc[4 * g + j].x);
        v[4 * j + 1] = __float_as_uint(acc[4 * g + j].y);
        v[4 * j + 2] = __float_as_uint(acc[4 * g + j].z);
        v[4 * j + 3] = __float_as_uint(acc[4 * g + j].w);
      }
      tmem_st16(lane_addr + col + h + 16 * g, v);
    }
  }
  tmem_st_wait();
}

// Sum of entry `i` of the vector parts (at D*D) of the state records p0 .. p1-1.
template <int D>
__device__ __forceinline__ float sum_vector_entry(const float* recs, long long stride, int p0, int p1, int i) {
  float acc = 0.f;
#pragma unroll 1
  for (int p = p0; p < p1; ++p) acc += recs[p * stride + D * D + i];
  return acc;
}

// The value a centred record set adds to row `row` of the held state: the
// sum of v over the records' tokens (entry D + row of the vector parts) for a
// row of S^T, `n_tok` (the records' token count) for a row of z (row == D).
template <int D>
__device__ __forceinline__ float centred_row_add(const float* recs, long long stride, int p0, int p1, int row,
                                                 float n_tok) {
  if (row < 0) return 0.f;
  return row < D ? sum_vector_entry<D>(recs, stride, p0, p1, D + row) : n_tok;
}

// Sum of the 8-entry slices [off, off + 8) of the vector parts (at D*D) of the
// state records p0 .. p1-1.
template <int D>
__device__ __forceinline__ void sum_vectors8(const float* recs, long long stride, int p0, int p1, int off,
                                             float (&acc)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 1
  for (int p = p0; p < p1; ++p) {
    const float4* src = reinterpret_cast<const float4*>(recs + p * stride + D * D + off);
    const float4 a = src[0], b = src[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
}

// The transpose of a D x D state held in tensor memory (this thread's lane is
// row `row` of the held matrix) to global memory, row-major: dst[c][row].
template <int D>
__device__ __forceinline__ void store_state_transposed(float* dst, uint32_t lane_addr, uint32_t col, int row) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(lane_addr + col + c0, v);
    tmem_ld_wait();
    if (row >= 0) {
#pragma unroll
      for (int j = 0; j < 32; ++j) dst[(long long)(c0 + j) * D + row] = __uint_as_float(v[j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult qr;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      (void)cudaGetLastError();
  }
  return fn;
}

// [BH][N][D] bf16 viewed as a 3-D tensor; boxes of [C rows][64 features],
// 128-byte swizzle, zero fill past the end of each sequence.
// [BH][N][D] bf16 tensor, boxes of 64 features x `rows` tokens, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* ptr, int BH, int N, int D, int rows = C) {
  auto enc = get_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace
}  // namespace la
