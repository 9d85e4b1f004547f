// Tensor-core (tcgen05) chunked causal forward for bf16 inputs, dk = dv = D in
// {64, 128}, chunks of C = 128 tokens.
//
// What one chunk computes (a re-association of the masked sums of
// "상태공간모델·선형 어텐션 — 어텐션의 O(N²) 대안", section 2, by the
// distributivity argument of "Linear Attention: KV를 고정 크기 상태에 누적하기",
// fig. 5; the state update is the recurrence of its section "상태 갱신과 읽기를
// 식으로 정리하기" applied to C tokens at once):
//   P    = phi(Q_c) phi(K_c)^T, masked to j <= t          (MMA1, TMEM fp32)
//   O    = phi(Q_c) S_prev + P V_c                         (MMA3 + MMA2)
//   den  = phi(Q_c) z_prev + P 1 + eps                     (CUDA cores, fp32)
//   S   += phi(K_c)^T V_c,  z += phi(K_c)^T 1              (MMA4; z on CUDA cores)
//   out  = O / den
// S lives in tensor memory in fp32 for the whole segment; its bf16 copy in
// shared memory is the B operand of MMA3.
//
// Two kernels share the machinery:
//   tc_state_kernel   per-segment sums dS = sum phi(k) v^T, dz = sum phi(k)
//   tc_forward_kernel the chunk loop above, starting from the segment's prefix
// (the CUDA-core scan kernel joins them). One CTA per (segment, b*h).
//
// Warp roles in tc_forward_kernel (320 threads):
//   warp 0      TMA producer: Q, K, V chunk tiles into a ring of stages
//   warp 1      TMEM allocator and MMA issuer (one elected lane)
//   warps 2-5   group A: phi in place on Q and K, z sums, S copy to smem
//   warps 6-9   group B: P mask/rowsum/bf16 pack, output epilogue
// Every wait is bounded; on a timeout the CTA sets the device status word,
// drains, frees its tensor memory and exits.
#include <cudaTypedefs.h>

#include "la_internal.cuh"
#include "la_sm100.cuh"

namespace la {

namespace {

using namespace sm100;

constexpr int C = 128;                    // tokens per chunk
constexpr int BOX = 128 * 128;            // bytes of one [128 rows][64 bf16] SW128 box
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int D>
struct Cfg {
  static constexpr int NB = D / 64;                   // 64-feature boxes per tile
  static constexpr int TILE = NB * BOX;               // one [C][D] bf16 tile
  static constexpr int ST = D == 128 ? 2 : 3;         // forward pipeline stages
  static constexpr int STAGE = 3 * TILE;              // Q, K, V
  static constexpr int SBUF = NB * D * 128;           // bf16 S copy, MN-major, D rows per box
  static constexpr int KSTEPS = D / 16;               // MMA k-steps over a head dimension
  // tensor memory columns
  static constexpr uint32_t COL_P0 = 0, COL_P1 = 128, COL_S = 256, COL_O = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  // state kernel
  static constexpr int ST_S = D == 128 ? 2 : 3;
  static constexpr int STAGE_S = 2 * TILE;            // K, V
  static constexpr uint32_t TMEM_COLS_S = D < 32 ? 32 : D;
};

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

// phi on 8 packed bf16 values in place; when `acc` is given, also add the
// unrounded fp32 phi values to it (column sums for z).
__device__ __forceinline__ void phi_bf16x8(uint4& w, float* acc) {
  uint32_t* p = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = phi_fast(__uint_as_float(p[i] << 16));
    const float hi = phi_fast(__uint_as_float(p[i] & 0xFFFF0000u));
    if (acc != nullptr) {
      acc[2 * i] += lo;
      acc[2 * i + 1] += hi;
    }
    p[i] = pack_bf16x2(lo, hi);
  }
}

__device__ __forceinline__ void report_timeout(int* status) { atomicExch(status, (int)LA_ERR_TIMEOUT); }

// Group A: phi in place on one [C][D] tile of stage memory; when `zacc` is
// given, also the column sums of phi over rows < n_valid (thread t owns
// logical 16-byte chunk t % 8 of each box and rows t/8 + 16 i).
template <int D>
__device__ __forceinline__ void phi_tile(uint8_t* tile, int t, int n_valid, float (*zacc)[8]) {
  constexpr int NB = D / 64;
  const int lc = t & 7, rg = t >> 3;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = rg + 16 * i;
      uint4* p = reinterpret_cast<uint4*>(tile + b * BOX + sw128(r, lc));
      uint4 w = *p;
      phi_bf16x8(w, (zacc != nullptr && r < n_valid) ? zacc[b] : nullptr);
      *p = w;
    }
  }
}

// Reduce the per-thread column partials of phi_tile across group A; thread f
// (< D) receives the column sum of feature f in *colsum. zsum: [D] floats,
// zero on entry and left zero on exit; zbar: an mbarrier of 128 arrivals used
// as the group's rendezvous (bounded, unlike bar.sync). Callers alternate two
// (zsum, zbar) pairs between chunks; `parity` is the pair's use count & 1.
template <int D>
__device__ __forceinline__ bool reduce_colsum(float (*zacc)[8], float* zsum, uint64_t* zbar, uint32_t parity,
                                              int t, volatile int* abort_flag, float* colsum) {
  constexpr int NB = D / 64;
  const int lane = t & 31, lc = t & 7;
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float x = zacc[b][e];
      x += __shfl_xor_sync(0xffffffffu, x, 8);
      x += __shfl_xor_sync(0xffffffffu, x, 16);
      if (lane < 8) atomicAdd(&zsum[b * 64 + lc * 8 + e], x);
    }
  mbar_arrive(zbar);
  if (!mbar_wait(zbar, parity, abort_flag, kTimeoutNs)) return false;
  float s = 0.f;
  if (t < D) {
    s = zsum[t];
    zsum[t] = 0.f;
  }
  *colsum = s;
  return true;
}

// Copy the fp32 state rows of this thread's TMEM lane to the bf16 MN-major
// operand buffer (row r = key component, 64 value columns per box).
template <int D>
__device__ __forceinline__ void copy_state_to_smem(uint32_t taddr_lane, uint8_t* sbuf, int row) {
  constexpr int NB = D / 64;
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(taddr_lane + c0, v);
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
  (void)NB;
}

template <int D>
struct FwdSmem {
  // stage ring, then the S operand; all boxes 1024-byte aligned
  static constexpr int OFF_STAGES = 0;
  static constexpr int OFF_SBUF = Cfg<D>::ST * Cfg<D>::STAGE;
  static constexpr int OFF_ZST = OFF_SBUF + Cfg<D>::SBUF;          // [ST][D] fp32
  static constexpr int OFF_ZSUM = OFF_ZST + Cfg<D>::ST * D * 4;    // [2][D] fp32
  static constexpr int OFF_BAR = OFF_ZSUM + 2 * D * 4;             // barriers
  static constexpr int NBAR = 3 * Cfg<D>::ST + 2 + 2 + 1 + 1 + 1 + 1 + 1 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
};

struct FwdParams {
  int N, P, seg_len;
  float eps;
  const float* ws_state;   // [BH][P][D*D + D] prefixes
  __nv_bfloat16* out;      // [BH][N][D]
  int* status;             // device status word (set on a bounded-wait timeout)
};

template <int D>
__global__ void __launch_bounds__(320, 1)
tc_forward_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const FwdParams prm) {
  using G = Cfg<D>;
  using L = FwdSmem<D>;
  constexpr int ST = G::ST;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sbuf = sm + L::OFF_SBUF;
  float* zst = reinterpret_cast<float*>(sm + L::OFF_ZST);
  float* zsum = reinterpret_cast<float*>(sm + L::OFF_ZSUM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* phi_done = bars + ST;
  uint64_t* empty = bars + 2 * ST;
  uint64_t* p_full = bars + 3 * ST;       // [2]
  uint64_t* p_ready = bars + 3 * ST + 2;  // [2]
  uint64_t* s_full = bars + 3 * ST + 4;
  uint64_t* s_ready = bars + 3 * ST + 5;
  uint64_t* o_full = bars + 3 * ST + 6;
  uint64_t* o_empty = bars + 3 * ST + 7;
  uint64_t* mma_fin = bars + 3 * ST + 8;
  uint64_t* zbar = bars + 3 * ST + 9;     // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::OFF_MISC + 4);
  // the swizzled operand boxes need 1024-byte alignment of the shared window
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
      mbar_init(&phi_done[i], 128);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_ready[i], 128);
    }
    mbar_init(s_full, 1);
    mbar_init(s_ready, 128);
    mbar_init(o_full, 1);
    mbar_init(o_empty, 128);
    mbar_init(mma_fin, 1);
    mbar_init(&zbar[0], 128);
    mbar_init(&zbar[1], 128);
    for (int i = 0; i < 2 * D; ++i) zsum[i] = 0.f;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % ST;
        if (c >= ST && !mbar_wait(&empty[s], ((c / ST) - 1) & 1, abort_flag, kTimeoutNs)) break;
        uint8_t* st = sm + s * G::STAGE;
        mbar_arrive_expect_tx(&full[s], 3 * G::TILE);
        const int y = tok0 + c * C;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) {
          tma_load_3d(st + b * BOX, &map_q, &full[s], 64 * b, y, bh);
          tma_load_3d(st + G::TILE + b * BOX, &map_k, &full[s], 64 * b, y, bh);
          tma_load_3d(st + 2 * G::TILE + b * BOX, &map_v, &full[s], 64 * b, y, bh);
        }
        issued = c + 1;
      }
      // drain: every issued load must land before the CTA's smem is released
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_wait(&full[c % ST], (c / ST) & 1, abort_flag, kTimeoutNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_qk = make_idesc_bf16(128, 128, false, false);   // P = phiQ phiK^T
      constexpr uint32_t id_qs = make_idesc_bf16(128, D, false, true);      // O = phiQ S
      constexpr uint32_t id_kv = make_idesc_bf16(D, D, true, true);         // S += phiK^T V
      constexpr uint32_t id_pv = make_idesc_bf16(128, D, false, true);      // O += P V
      const uint32_t sbuf_a = smem_u32(sbuf);
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST;
        const uint32_t qa = smem_u32(sm + s * G::STAGE);
        const uint32_t ka = qa + G::TILE;
        const uint32_t va = qa + 2 * G::TILE;
        const uint32_t pcol = (c & 1) ? G::COL_P1 : G::COL_P0;
        ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(tmem + pcol, make_sdesc(qa + off, 16, 1024, kSwizzle128B),
                 make_sdesc(ka + off, 16, 1024, kSwizzle128B), id_qk, k > 0);
        }
        tc_commit(&p_full[c & 1]);
        ok = mbar_wait(s_ready, c & 1, abort_flag, kTimeoutNs);
        if (ok && c > 0) ok = mbar_wait(o_empty, (c - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(tmem + G::COL_O, make_sdesc(qa + off, 16, 1024, kSwizzle128B),
                 make_sdesc(sbuf_a + k * 2048, D * 128, 1024, kSwizzle128B), id_qs, k > 0);
        }
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ss(tmem + G::COL_S, make_sdesc(ka + k * 2048, BOX, 1024, kSwizzle128B),
                 make_sdesc(va + k * 2048, BOX, 1024, kSwizzle128B), id_kv, 1);
        tc_commit(s_full);
        ok = mbar_wait(&p_ready[c & 1], (c >> 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ts(tmem + G::COL_O, tmem + pcol + k * 8, make_sdesc(va + k * 2048, BOX, 1024, kSwizzle128B),
                 id_pv, 1);
        tc_commit(o_full);
        tc_commit(&empty[s]);
      }
      // every MMA issued must have finished before tensor memory is released
      tc_commit(mma_fin);
      mbar_wait(mma_fin, 0, abort_flag, kTimeoutNs);
    }
  } else if (warp < 6) {
    // ---------------- group A: phi, z, state copy ----------------
    const int t = tid - 64;                 // 0..127
    const int q = warp & 3;                 // TMEM quadrant of this warp
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    // initial state: prefix of this segment, into TMEM (fp32) lanes
    const float* st = prm.ws_state + ((long long)bh * prm.P + seg) * (long long)(D * D + D);
    float zrun = (t < D) ? st[D * D + t] : 0.f;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 16) {
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = row >= 0 ? __float_as_uint(st[row * D + c0 + j]) : 0u;
      tmem_st16(lane_addr + G::COL_S + c0, v);
    }
    tmem_st_wait();
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      uint8_t* stg = sm + s * G::STAGE;
      const int n_valid = min(C, tok_end - (tok0 + c * C));
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      float zacc[G::NB][8];
#pragma unroll
      for (int b = 0; b < G::NB; ++b)
#pragma unroll
        for (int e = 0; e < 8; ++e) zacc[b][e] = 0.f;
      phi_tile<D>(stg, t, C, nullptr);            // Q
      phi_tile<D>(stg + G::TILE, t, n_valid, zacc);  // K, with column sums
      float colsum = 0.f;
      ok = reduce_colsum<D>(zacc, zsum + (c & 1) * D, &zbar[c & 1], (c >> 1) & 1, t, abort_flag, &colsum);
      if (!ok) break;
      if (t < D) {
        zst[s * D + t] = zrun;  // z before this chunk, for group B's denominators
        zrun += colsum;
      }
      fence_proxy_async_smem();
      mbar_arrive(&phi_done[s]);
      // bf16 copy of the state before this chunk (after the previous update)
      if (c > 0) {
        ok = mbar_wait(s_full, (c - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
      }
      copy_state_to_smem<D>(lane_addr + G::COL_S, sbuf, row);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(s_ready);
    }
  } else {
    // ---------------- group B: P and the output epilogue ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;            // chunk row (query token) of this thread
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    __nv_bfloat16* outb = prm.out + (long long)bh * prm.N * D;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      const uint8_t* qt = sm + s * G::STAGE;
      const uint32_t pcol = (c & 1) ? G::COL_P1 : G::COL_P0;
      ok = mbar_wait(&p_full[c & 1], (c >> 1) & 1, abort_flag, kTimeoutNs) &&
           mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      // masked P row: fp32 row sum, bf16 pack back into the first 64 columns
      float rowsum = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < C; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(lane_addr + pcol + c0, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float a = (c0 + 2 * j <= r) ? __uint_as_float(v[2 * j]) : 0.f;
          const float b = (c0 + 2 * j + 1 <= r) ? __uint_as_float(v[2 * j + 1]) : 0.f;
          rowsum += a + b;
          pk[j] = pack_bf16x2(a, b);
        }
        tmem_st16(lane_addr + pcol + c0 / 2, pk);
      }
      // phi(q_r) . z_prev from the phi-transformed Q tile (swizzled rows)
      float dot = 0.f;
      const float* zp = zst + s * D;
#pragma unroll
      for (int b = 0; b < G::NB; ++b)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 w = *reinterpret_cast<const uint4*>(qt + b * BOX + sw128(r, ch));
          const uint32_t* p = reinterpret_cast<const uint32_t*>(&w);
          const int f = b * 64 + ch * 8;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dot = fmaf(__uint_as_float(p[i] << 16), zp[f + 2 * i], dot);
            dot = fmaf(__uint_as_float(p[i] & 0xFFFF0000u), zp[f + 2 * i + 1], dot);
          }
        }
      const float inv_den = 1.f / (rowsum + dot + prm.eps);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_ready[c & 1]);
      // output rows
      ok = mbar_wait(o_full, c & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      const int tok = tok0 + c * C + r;
      uint4* dst = reinterpret_cast<uint4*>(outb + (long long)tok * D);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(lane_addr + G::COL_O + c0, v);
        tmem_ld_wait();
        if (tok < tok_end) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * inv_den, __uint_as_float(v[8 * j + 1]) * inv_den);
            w.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv_den, __uint_as_float(v[8 * j + 3]) * inv_den);
            w.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv_den, __uint_as_float(v[8 * j + 5]) * inv_den);
            w.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv_den, __uint_as_float(v[8 * j + 7]) * inv_den);
            dst[c0 / 8 + j] = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(o_empty);
    }
  }

  // ---------------- teardown ----------------
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Per-segment state sums: dS = phi(K_seg)^T V_seg (tensor cores, fp32 in
// TMEM), dz = column sums of phi(K_seg) (CUDA cores). 192 threads:
// warp 0 TMA, warp 1 MMA, warps 2-5 phi + z + final store.
// ---------------------------------------------------------------------------
template <int D>
struct StateSmem {
  static constexpr int OFF_ZSUM = Cfg<D>::ST_S * Cfg<D>::STAGE_S;
  static constexpr int OFF_BAR = OFF_ZSUM + 2 * D * 4;
  static constexpr int NBAR = 3 * Cfg<D>::ST_S + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
};

struct StateParams {
  int N, P, seg_len;
  float* ws_state;  // [BH][P][D*D + D]
  int* status;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                const StateParams prm) {
  using G = Cfg<D>;
  using L = StateSmem<D>;
  constexpr int ST = G::ST_S;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  float* zsum = reinterpret_cast<float*>(sm + L::OFF_ZSUM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* phi_done = bars + ST;
  uint64_t* empty = bars + 2 * ST;
  uint64_t* s_full = bars + 3 * ST;
  uint64_t* mma_fin = bars + 3 * ST + 1;
  uint64_t* zbar = bars + 3 * ST + 2;     // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::OFF_MISC + 4);
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
      mbar_init(&phi_done[i], 128);
      mbar_init(&empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(mma_fin, 1);
    mbar_init(&zbar[0], 128);
    mbar_init(&zbar[1], 128);
    for (int i = 0; i < 2 * D; ++i) zsum[i] = 0.f;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, G::TMEM_COLS_S);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % ST;
        if (c >= ST && !mbar_wait(&empty[s], ((c / ST) - 1) & 1, abort_flag, kTimeoutNs)) break;
        uint8_t* st = sm + s * G::STAGE_S;
        mbar_arrive_expect_tx(&full[s], 2 * G::TILE);
        const int y = tok0 + c * C;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) {
          tma_load_3d(st + b * BOX, &map_k, &full[s], 64 * b, y, bh);
          tma_load_3d(st + G::TILE + b * BOX, &map_v, &full[s], 64 * b, y, bh);
        }
        issued = c + 1;
      }
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_wait(&full[c % ST], (c / ST) & 1, abort_flag, kTimeoutNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_kv = make_idesc_bf16(D, D, true, true);
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % ST;
        const uint32_t ka = smem_u32(sm + s * G::STAGE_S);
        const uint32_t va = ka + G::TILE;
        ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ss(tmem, make_sdesc(ka + k * 2048, BOX, 1024, kSwizzle128B),
                 make_sdesc(va + k * 2048, BOX, 1024, kSwizzle128B), id_kv, (c > 0 || k > 0) ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      tc_commit(s_full);
      tc_commit(mma_fin);
      mbar_wait(mma_fin, 0, abort_flag, kTimeoutNs);
    }
  } else {
    const int t = tid - 64;
    const int q = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    float zrun = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      uint8_t* stg = sm + s * G::STAGE_S;
      const int n_valid = min(C, tok_end - (tok0 + c * C));
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      float zacc[G::NB][8];
#pragma unroll
      for (int b = 0; b < G::NB; ++b)
#pragma unroll
        for (int e = 0; e < 8; ++e) zacc[b][e] = 0.f;
      phi_tile<D>(stg, t, n_valid, zacc);
      float colsum = 0.f;
      ok = reduce_colsum<D>(zacc, zsum + (c & 1) * D, &zbar[c & 1], (c >> 1) & 1, t, abort_flag, &colsum);
      if (!ok) break;
      zrun += colsum;
      fence_proxy_async_smem();
      mbar_arrive(&phi_done[s]);
    }
    float* dst = prm.ws_state + ((long long)bh * prm.P + seg) * (long long)(D * D + D);
    if (ok) ok = mbar_wait(s_full, 0, abort_flag, kTimeoutNs);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(lane_addr + c0, v);
        tmem_ld_wait();
        if (row >= 0) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + row * D + c0 + j) =
                make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                            __uint_as_float(v[j + 3]));
        }
      }
      if (t < D) dst[D * D + t] = zrun;
    }
  }
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS_S);
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
cudaError_t make_map(CUtensorMap* m, const void* ptr, int BH, int N, int D) {
  auto enc = get_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)C, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_state(const FwdArgs& a) {
  CUtensorMap mk, mv;
  cudaError_t e = make_map(&mk, a.k, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mv, a.v, a.BH, a.N, D);
  if (e != cudaSuccess) return e;
  constexpr int smem = StateSmem<D>::BYTES;
  e = cudaFuncSetAttribute(tc_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  StateParams p{a.N, a.plan.P, a.plan.seg_len, a.ws_state, device_status_ptr()};
  tc_state_kernel<D><<<a.BH * a.plan.P, 192, smem, a.stream>>>(mk, mv, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <int D>
cudaError_t launch_forward(const FwdArgs& a) {
  CUtensorMap mq, mk, mv;
  cudaError_t e = make_map(&mq, a.q, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mk, a.k, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mv, a.v, a.BH, a.N, D);
  if (e != cudaSuccess) return e;
  constexpr int smem = FwdSmem<D>::BYTES;
  static_assert(smem <= 232448, "shared memory budget");
  e = cudaFuncSetAttribute(tc_forward_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  FwdParams p{a.N, a.plan.P, a.plan.seg_len, a.eps, a.ws_state, (__nv_bfloat16*)a.out, device_status_ptr()};
  tc_forward_kernel<D><<<a.BH * a.plan.P, 320, smem, a.stream>>>(mq, mk, mv, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace

bool tc_forward_supported(int dk, int dv, la_dtype dtype, int causal) {
  return dtype == LA_BF16 && dk == dv && (dk == 64 || dk == 128) && causal;
}

cudaError_t tc_segment_state(const FwdArgs& a) {
  return a.dk == 128 ? launch_state<128>(a) : launch_state<64>(a);
}

cudaError_t tc_forward_output(const FwdArgs& a) {
  return a.dk == 128 ? launch_forward<128>(a) : launch_forward<64>(a);
}

}  // namespace la
