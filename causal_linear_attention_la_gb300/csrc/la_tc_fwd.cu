// Tensor-core (tcgen05) chunked causal forward for bf16 inputs, dk = dv = D in
// {64, 128}, chunks of C = 128 tokens.
//
// What one chunk computes (a re-association of the masked sums of
// "상태공간모델·선형 어텐션 — 어텐션의 O(N²) 대안", section 2, by the
// distributivity argument of "Linear Attention: KV를 고정 크기 상태에 누적하기",
// fig. 5; the state update is the recurrence of its section "상태 갱신과 읽기를
// 식으로 정리하기" applied to C tokens at once):
//   P    = phi(Q_c) phi(K_c)^T, masked to j <= t            MMA1 (tensor cores)
//   O    = phi(Q_c) S_prev + P V_c                           MMA3, MMA2
//   S   += phi(K_c)^T V_c                                    MMA4
//   z   += column sums of phi(K_c)                           CUDA cores, fp32
//   den  = phi(Q_c) z_prev + P 1 + eps                       CUDA cores, fp32
//   out  = O / den
// S lives in tensor memory in fp32 for the whole segment; its bf16 copy in
// shared memory is the B operand of MMA3. The normaliser terms stay on the
// CUDA cores: measured on GB300, a thin (N = 16) tcgen05.mma costs nearly as
// much as a full-width one, while the row and column sums fall out of passes
// the CUDA cores make anyway.
//
// Two kernels share the machinery:
//   tc_state_kernel   per-segment sums dS = sum phi(k) v^T, dz = sum phi(k)
//   tc_forward_kernel the chunk loop above, starting from the segment's prefix
// (the scan kernel joins them). One CTA per (segment, b*h).
//
// Warp roles in tc_forward_kernel (448 threads):
//   warps 0-3    group C: phi in place on K with the column sums that update z
//   warps 4-7    group A: phi in place on Q; state copy S -> shared memory
//   warps 8-11   group B: P mask, bf16 pack and row sums; denominators; epilogue
//   warp 12      TMA producer: Q, K, V chunk tiles into a ring of stages
//   warp 13      TMEM allocator and MMA issuer (one elected lane)
// (the CUDA-core groups take the lowest warp ids, which the warp schedulers
// favour; each group's four warps cover the four TMEM lane quadrants)
// phi(K) is rounded to nearest from an fp32 exponential, since z is summed
// from it; phi(Q) uses packed bf16 arithmetic (a common scale error of
// phi(q) cancels between numerator and denominator).
// Every wait is bounded; on a timeout the CTA sets the device status word,
// drains, frees its tensor memory and exits.
#include "la_tc_common.cuh"

namespace la {

namespace {

using namespace sm100;

template <int D>
struct Cfg {
  static constexpr int NB = D / 64;                   // 64-feature boxes per tile
  static constexpr int TILE = NB * BOX;               // one [C][D] bf16 tile
  static constexpr int ST = D == 128 ? 2 : 3;         // forward pipeline stages
  static constexpr int STAGE = 3 * TILE;              // Q, K, V
  static constexpr int SBUF = NB * D * 128;           // bf16 S copy, MN-major, D rows per box
  static constexpr int KSTEPS = D / 16;               // MMA k-steps over a head dimension
  static constexpr int NPB = 2;                       // P buffers in tensor memory
  // tensor memory columns
  static constexpr uint32_t COL_P = 0;                // NPB x 128
  static constexpr uint32_t COL_S = 128 * NPB;        // D
  static constexpr uint32_t COL_O = COL_S + D;        // D
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_O + D <= TMEM_COLS, "tensor memory budget");
  // state kernel
  static constexpr int ST_S = D == 128 ? 2 : 3;
  static constexpr int STAGE_S = 2 * TILE;            // K, V
  static constexpr uint32_t TMEM_COLS_S = D == 128 ? 128 : 64;
};

template <int D>
struct FwdSmem {
  static constexpr int OFF_SBUF = Cfg<D>::ST * Cfg<D>::STAGE;      // all boxes 1024-aligned
  static constexpr int OFF_ZST = OFF_SBUF + Cfg<D>::SBUF;          // [ST][D] fp32: z before each staged chunk
  static constexpr int OFF_BAR = OFF_ZST + Cfg<D>::ST * D * 4;
  static constexpr int NBAR = 3 * Cfg<D>::ST + 2 * Cfg<D>::NPB + 5;
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
__global__ void __launch_bounds__(448, 1)
tc_forward_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const FwdParams prm) {
  using G = Cfg<D>;
  using L = FwdSmem<D>;
  constexpr int ST = G::ST, NPB = G::NPB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sbuf = sm + L::OFF_SBUF;
  float* zst = reinterpret_cast<float*>(sm + L::OFF_ZST);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* phi_done = bars + ST;
  uint64_t* empty = bars + 2 * ST;
  uint64_t* p_full = bars + 3 * ST;              // [NPB]
  uint64_t* p_ready = bars + 3 * ST + NPB;       // [NPB]
  uint64_t* s_full = bars + 3 * ST + 2 * NPB;
  uint64_t* s_ready = s_full + 1;
  uint64_t* o_full = s_full + 2;
  uint64_t* o_empty = s_full + 3;
  uint64_t* mma_fin = s_full + 4;
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
  const float* st = prm.ws_state + ((long long)bh * prm.P + seg) * (long long)(D * D + D);

  if (tid == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&phi_done[i], 256);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < NPB; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_ready[i], 128);
    }
    mbar_init(s_full, 1);
    mbar_init(s_ready, 128);
    mbar_init(o_full, 1);
    mbar_init(o_empty, 128);
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
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % ST;
        if (c >= ST && !mbar_wait(&empty[s], ((c / ST) - 1) & 1, abort_flag, kTimeoutNs)) break;
        uint8_t* stg = sm + s * G::STAGE;
        mbar_arrive_expect_tx(&full[s], 3 * G::TILE);
        const int y = tok0 + c * C;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) {
          tma_load_3d(stg + b * BOX, &map_q, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + G::TILE + b * BOX, &map_k, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + 2 * G::TILE + b * BOX, &map_v, &full[s], 64 * b, y, bh);
        }
        issued = c + 1;
      }
      // drain: every issued load must land before the CTA's smem is released
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_wait(&full[c % ST], (c / ST) & 1, abort_flag, kTimeoutNs);
    }
  } else if (warp == 13) {
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
        const int pb = c % NPB;
        const uint32_t pcol = G::COL_P + 128 * pb;
        ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(tmem + pcol, make_sdesc(qa + off, 16, 1024, kSwizzle128B),
                 make_sdesc(ka + off, 16, 1024, kSwizzle128B), id_qk, k > 0);
        }
        tc_commit(&p_full[pb]);
        ok = mbar_wait(s_ready, c & 1, abort_flag, kTimeoutNs);
        if (ok && c > 0) ok = mbar_wait(o_empty, (c - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k)
          mma_ss(tmem + G::COL_O, make_sdesc(qa + (k >> 2) * BOX + (k & 3) * 32, 16, 1024, kSwizzle128B),
                 make_sdesc(sbuf_a + k * 2048, D * 128, 1024, kSwizzle128B), id_qs, k > 0);
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ss(tmem + G::COL_S, make_sdesc(ka + k * 2048, BOX, 1024, kSwizzle128B),
                 make_sdesc(va + k * 2048, BOX, 1024, kSwizzle128B), id_kv, 1);
        tc_commit(s_full);
        ok = mbar_wait(&p_ready[pb], (c / NPB) & 1, abort_flag, kTimeoutNs);
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
  } else if (warp >= 4 && warp < 8) {
    // ---------------- group A: phi(Q), state copy ----------------
    const int t = tid - 128;                // 0..127
    const int q = warp & 3;                 // TMEM quadrant of this warp
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    // initial state (this segment's prefix) into TMEM
    const float4* srow = reinterpret_cast<const float4*>(st + (row >= 0 ? row : 0) * D);
#pragma unroll
    for (int h = 0; h < D; h += 64) {        // 64 columns per batch: 16 loads in flight
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
        tmem_st16(lane_addr + G::COL_S + h + 16 * g, v);
      }
    }
    tmem_st_wait();
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      phi_tile_bf16<D, 128>(sm + s * G::STAGE, t);   // Q
      fence_proxy_async_smem();
      mbar_arrive(&phi_done[s]);
      // bf16 copy of the state before chunk c (after the previous update)
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
  } else if (warp >= 8 && warp < 12) {
    // ---------------- group B: P, denominators and the output epilogue ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;            // chunk row (query token) of this thread
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    __nv_bfloat16* outb = prm.out + (long long)bh * prm.N * D;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      const int pb = c % NPB;
      const uint32_t pcol = G::COL_P + 128 * pb;
      ok = mbar_wait(&p_full[pb], (c / NPB) & 1, abort_flag, kTimeoutNs) &&
           mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      // masked P row in bf16, packed into the first 64 columns of its buffer,
      // and its fp32 row sum. Warp q holds rows 32q..32q+31: 32-column pieces
      // left of q are kept whole, piece q is masked per lane, pieces right of
      // q are zero.
      float rowsum = 0.f;
#pragma unroll 1
      for (int p = 0; p < 4; ++p) {
        uint32_t pk[16];
        if (p <= q) {
          uint32_t v[32];
          tmem_ld32(lane_addr + pcol + 32 * p, v);
          tmem_ld_wait();
          const int lim = p < q ? 32 : (r - 32 * p + 1);  // columns kept in this piece
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a = (2 * j < lim) ? __uint_as_float(v[2 * j]) : 0.f;
            const float b = (2 * j + 1 < lim) ? __uint_as_float(v[2 * j + 1]) : 0.f;
            rowsum += a + b;
            pk[j] = pack_bf16x2(a, b);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = 0u;
        }
        tmem_st16(lane_addr + pcol + 16 * p, pk);
      }
      // phi(q_r) . z_prev from the phi-transformed Q tile (swizzled rows)
      float dot = 0.f;
      {
        const uint8_t* qt = sm + s * G::STAGE;
        const float* zp = zst + s * D;
#pragma unroll 1
        for (int b = 0; b < G::NB; ++b)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 w = *reinterpret_cast<const uint4*>(qt + b * BOX + sw128(r, ch));
            const uint32_t* pw = reinterpret_cast<const uint32_t*>(&w);
            const float4 z0 = *reinterpret_cast<const float4*>(zp + b * 64 + ch * 8);
            const float4 z1 = *reinterpret_cast<const float4*>(zp + b * 64 + ch * 8 + 4);
            dot = fmaf(__uint_as_float(pw[0] << 16), z0.x, dot);
            dot = fmaf(__uint_as_float(pw[0] & 0xFFFF0000u), z0.y, dot);
            dot = fmaf(__uint_as_float(pw[1] << 16), z0.z, dot);
            dot = fmaf(__uint_as_float(pw[1] & 0xFFFF0000u), z0.w, dot);
            dot = fmaf(__uint_as_float(pw[2] << 16), z1.x, dot);
            dot = fmaf(__uint_as_float(pw[2] & 0xFFFF0000u), z1.y, dot);
            dot = fmaf(__uint_as_float(pw[3] << 16), z1.z, dot);
            dot = fmaf(__uint_as_float(pw[3] & 0xFFFF0000u), z1.w, dot);
          }
      }
      const float inv_den = 1.f / (rowsum + dot + prm.eps);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_ready[pb]);
      // output rows
      ok = mbar_wait(o_full, c & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      const int tok = tok0 + c * C + r;
      uint4* dst = reinterpret_cast<uint4*>(outb + (long long)tok * D);
#pragma unroll 1
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
  } else {
    // ---------------- group C: phi(K) and z ----------------
    using X = ExactLayout<D, 128>;
    const int t = tid;                      // 0..127
    const int fc = X::FCW * (t >> 5) + (lane % X::FCW);
    const bool owner = lane < X::FCW;       // holds the z of features 8 fc .. 8 fc + 7
    float zrun[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) zrun[e] = owner ? st[D * D + 8 * fc + e] : 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      const int n_valid = min(C, tok_end - (tok0 + c * C));
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      float colsum[8];
      phi_tile_exact<D, 128>(sm + s * G::STAGE + G::TILE, t, n_valid, colsum);  // K
      fence_proxy_async_smem();
      if (owner) {
        // z before this chunk, for group B's denominators
        float4* zd = reinterpret_cast<float4*>(zst + s * D + 8 * fc);
        zd[0] = make_float4(zrun[0], zrun[1], zrun[2], zrun[3]);
        zd[1] = make_float4(zrun[4], zrun[5], zrun[6], zrun[7]);
#pragma unroll
        for (int e = 0; e < 8; ++e) zrun[e] += colsum[e];
      }
      mbar_arrive(&phi_done[s]);
    }
  }

  // ---------------- teardown ----------------
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Per-segment state sums: dS = phi(K_seg)^T V_seg on the tensor cores into
// TMEM (fp32), dz = column sums of phi(K_seg) on the CUDA cores (fp32).
// 320 threads: warps 0-7 phi(K) (rounded to nearest) and z, warps 0-3 also
// the final store of dS; warp 8 TMA, warp 9 TMEM allocator and MMA.
// ---------------------------------------------------------------------------
template <int D>
struct StateSmem {
  static constexpr int OFF_BAR = Cfg<D>::ST_S * Cfg<D>::STAGE_S;
  static constexpr int NBAR = 3 * Cfg<D>::ST_S + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
};

struct StateParams {
  int N, P, seg_len;
  float* ws_state;  // [BH][P][D*D + D]
  int* status;
};

template <int D>
__global__ void __launch_bounds__(320, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                const StateParams prm) {
  using G = Cfg<D>;
  using L = StateSmem<D>;
  constexpr int ST = G::ST_S;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* phi_done = bars + ST;
  uint64_t* empty = bars + 2 * ST;
  uint64_t* s_full = bars + 3 * ST;
  uint64_t* mma_fin = bars + 3 * ST + 1;
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
      mbar_init(&phi_done[i], 256);
      mbar_init(&empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(mma_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, G::TMEM_COLS_S);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    if (lane == 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % ST;
        if (c >= ST && !mbar_wait(&empty[s], ((c / ST) - 1) & 1, abort_flag, kTimeoutNs)) break;
        uint8_t* stg = sm + s * G::STAGE_S;
        mbar_arrive_expect_tx(&full[s], 2 * G::TILE);
        const int y = tok0 + c * C;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) {
          tma_load_3d(stg + b * BOX, &map_k, &full[s], 64 * b, y, bh);
          tma_load_3d(stg + G::TILE + b * BOX, &map_v, &full[s], 64 * b, y, bh);
        }
        issued = c + 1;
      }
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_wait(&full[c % ST], (c / ST) & 1, abort_flag, kTimeoutNs);
    }
  } else if (warp == 9) {
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
    using X = ExactLayout<D, 256>;
    const int t = tid;                      // 0..255
    const int q = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    const int fc = X::FCW * (t >> 5) + (lane % X::FCW);
    float zrun[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) zrun[e] = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      const int n_valid = min(C, tok_end - (tok0 + c * C));
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      float colsum[8];
      phi_tile_exact<D, 256>(sm + s * G::STAGE_S, t, n_valid, colsum);
      fence_proxy_async_smem();
      mbar_arrive(&phi_done[s]);
#pragma unroll
      for (int e = 0; e < 8; ++e) zrun[e] += colsum[e];
    }
    float* dst = prm.ws_state + ((long long)bh * prm.P + seg) * (long long)(D * D + D);
    if (ok && lane < X::FCW) {
      float4* zd = reinterpret_cast<float4*>(dst + D * D + 8 * fc);
      zd[0] = make_float4(zrun[0], zrun[1], zrun[2], zrun[3]);
      zd[1] = make_float4(zrun[4], zrun[5], zrun[6], zrun[7]);
    }
    if (ok && warp < 4) ok = mbar_wait(s_full, 0, abort_flag, kTimeoutNs);
    if (ok && warp < 4) {
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
    }
  }
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS_S);
  }
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
  tc_state_kernel<D><<<a.BH * a.plan.P, 320, smem, a.stream>>>(mk, mv, p);
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
  tc_forward_kernel<D><<<a.BH * a.plan.P, 448, smem, a.stream>>>(mq, mk, mv, p);
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
