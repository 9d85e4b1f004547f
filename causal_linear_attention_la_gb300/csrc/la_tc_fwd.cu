// Tensor-core (tcgen05) chunked forward for bf16 inputs, dk = dv = D in
// {64, 128}, chunks of C = 128 tokens: causal, and non-causal (every query
// reads the whole sequence's state; tc_noncausal_kernel below).
//
// What one chunk computes (a re-association of the masked sums of
// "상태공간모델·선형 어텐션 — 어텐션의 O(N²) 대안", section 2, by the
// distributivity argument of "Linear Attention: KV를 고정 크기 상태에 누적하기",
// fig. 5; the state update is the recurrence of its section "상태 갱신과 읽기를
// 식으로 정리하기" applied to C tokens at once):
//   P    = phi(Q_c) phi(K_c)^T, masked to j <= t            tensor cores
//   O    = phi(Q_c) S_prev + P V_c                           tensor cores
//   S   += phi(K_c)^T V_c                                    tensor cores
//   z   += column sums of phi(K_c)
//   den  = phi(Q_c) z_prev + P 1 + eps
//   out  = O / den
// The state is held transposed (S^T, value index first) in fp32 tensor
// memory for the whole segment: S^T += V^T phi(K) reads both tiles as they
// arrive, and its bf16 copy in shared memory is then a K-major operand. At
// D = 64 the normaliser rides in the MMAs too (on GB300 an MMA instruction
// costs about the same for any N up to 256, so fewer, wider instructions are
// faster): the copy [S^T ; z rows] sits right after the K tile, so P,
// phi(Q) S_prev and phi(Q) z_prev come out of one N = 208 MMA; P V runs on
// [V | 1], so P 1 comes with it; and the held state is [S^T ; z] with a block
// of ones under V^T, so z is updated by the state MMA. At D = 128 z and den
// are summed on the CUDA cores, in fp32, in passes they make anyway.
//
// Two kernels:
//   tc_state_kernel   per-segment sums dS^T = V^T phi(K), dz = sum phi(k), for
//                     every segment but the last of each sequence (causal) or
//                     for all of them (non-causal)
//   tc_forward_kernel the chunk loop above; it starts from the sum of the
//                     records of the earlier segments (the exclusive prefix),
//                     and the last segment writes the final state.
// One CTA per (segment, b*h). The forward kernel is launched as a dependent
// of the state kernel: it fills its pipeline before waiting for the records.
//
// Warp roles in tc_forward_kernel (448 threads):
//   warps 0-3    group C: phi in place on K (with the column sums that
//                update z at D = 128)
//   warps 4-7    group A: phi in place on Q; state copy S^T -> shared memory
//   warps 8-11   group B: P mask and bf16 pack (row sums at D = 128);
//                denominators; epilogue
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
  static constexpr int SBUF = NB * D * 128;           // bf16 copy of S^T, D rows per box
  static constexpr bool MERGE = D == 64;              // P, phi(Q) S_prev and phi(Q) z_prev in one MMA
  static constexpr int ST = D == 64 ? 3 : 2;          // forward pipeline stages
  // MERGE: the state is held as one M = 128 accumulator [S^T ; z ... z]
  // (lanes 0..D-1 the rows of S^T, lanes D..127 copies of z), and its bf16
  // copy (D rows of S^T, then ZR rows of z) follows the K tile, so that one
  // MMA with N = 128 + D + ZR gives [P | phi(Q) S_prev | phi(Q) z_prev].
  static constexpr int ZR = 16;                       // z rows in the copy (N granule)
  static constexpr int NQK = MERGE ? 128 + D + ZR : 128;
  static constexpr int SBM = (D + ZR) * 128;          // MERGE: bytes of the copy
  // stage layout: Q, K, [S^T and z copy if MERGE], V
  static constexpr int OFF_K = TILE;
  static constexpr int OFF_SB = 2 * TILE;             // MERGE only: rows 128.. of the K operand
  static constexpr int OFF_V = MERGE ? 2 * TILE + SBM : 2 * TILE;
  static constexpr int STAGE = OFF_V + TILE;
  static_assert(OFF_V % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static constexpr int KSTEPS = D / 16;               // MMA k-steps over a head dimension
  static constexpr int NPB = 2;                       // P buffers in tensor memory
  static constexpr int NOB = MERGE ? 2 : 1;           // O buffers (each follows its P when MERGE)
  // tensor memory columns; MERGE: per buffer [P 128 | O D | den ZR], 224 apart
  __host__ __device__ static constexpr uint32_t pcol(int pb) { return MERGE ? pb * 224 : 128 * pb; }
  __host__ __device__ static constexpr uint32_t ocol(int ob) { return MERGE ? ob * 224 + 128 : 128 * NPB + D; }
  static constexpr uint32_t COL_S = MERGE ? 448 : 128 * NPB;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_S + D <= TMEM_COLS && ocol(NOB - 1) + D <= TMEM_COLS, "tensor memory budget");
  // state kernel
  static constexpr int ST_S = D == 128 ? 3 : 6;    // state-pass stages (bytes in flight hide DRAM latency)
  static constexpr int STAGE_S = 2 * TILE;            // K, V
  static constexpr uint32_t TMEM_COLS_S = 128;
};

template <int D>
struct FwdSmem {
  using G = Cfg<D>;
  // MERGE: a [C][64] tile of bf16 ones, the second 64-wide block of the V
  // operands: rows D.. of V^T (so the state MMA also sums z) and columns D..
  // of [V | 1] (so P V also sums the rows of P)
  static constexpr int OFF_ONES = G::ST * G::STAGE;
  // MERGE: two output tiles; each warp of group B stores its 32 rows with TMA,
  // so a stage is free as soon as its chunk's MMAs are done (!MERGE: the
  // output is staged in the chunk's Q tile and stored by the producer)
  static constexpr int OFF_OUT = OFF_ONES + (G::MERGE ? BOX : 0);
  static constexpr int OFF_SBUF = OFF_OUT + (G::MERGE ? 2 * G::TILE : 0);  // !MERGE: the S^T copy (1024-aligned)
  static constexpr int OFF_ZST = OFF_SBUF + (G::MERGE ? 0 : G::SBUF);  // !MERGE: [ST][D] fp32 z before each staged chunk
  static constexpr int OFF_BAR = OFF_ZST + (G::MERGE ? 0 : G::ST * D * 4);
  static constexpr int NBAR = 4 * G::ST + 2 * G::NPB + 2 * G::NOB + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

struct FwdParams {
  int N, P, seg_len, F;
  float eps;
  const float* ws_state;   // [BH][P*F][rec_words] sums over each state-pass part (segments 0..P-2)
  __nv_bfloat16* out;      // [BH][N][D]
  float* S_final;          // [BH][D][D] or null (written by the last segment)
  float* z_final;          // [BH][D] or null
  int* status;             // device status word (set on a bounded-wait timeout)
  // decay gating (the kDecay kernels): per-head factors and the state-pass part length
  const float* alpha = nullptr;   // [H]
  int H = 1;
  int sub_len = 0;
  // test of the bounded waits: the MMA issuer first waits on a barrier that
  // nothing completes (la_test_timeout_next_forward)
  int timeout_test = 0;
  // balanced pieces (SegPlan, d = 128 causal without a final state): CTA i
  // runs chunks i * piece_len .. of the heads laid end to end
  int NP = 0, piece_len = 0, nch = 0, BH = 0;
};

// The chunks one CTA of the chunk loop runs. By segments: chunks of head bh
// from token tok0. By pieces: global chunks g0, g0 + 1, ... of the heads
// laid end to end (nch chunks each), so a piece may end one head and start
// the next; chunk c then belongs to head (g0 + c) / nch.
struct ChunkMap {
  long long g0;
  int nch, bh, tok0, N;
  bool pieces;
  __device__ __forceinline__ int bh_of(int c) const { return pieces ? (int)((g0 + c) / nch) : bh; }
  __device__ __forceinline__ int y_of(int c) const {
    return pieces ? (int)((g0 + c) % nch) * C : tok0 + c * C;
  }
  // chunk c > 0 starts a head: the state goes back to zero
  __device__ __forceinline__ bool head_start(int c) const { return pieces && c > 0 && (g0 + c) % nch == 0; }
  __device__ __forceinline__ int n_valid(int c) const { return min(C, N - y_of(c)); }
};

// With decay gating (kDecay, D = 64): S_t = a S_{t-1} + phi(k_t) v_t^T and the
// same for z ("Linear Attention, 곱의 순서를 바꾸면 생기는 일", paragraph on 감쇠
// 게이팅). For a chunk of n tokens starting from S_prev:
//   row r reads a^(r+1) S_prev: phi(Q) rows are weighted a^(r+1);
//   token j enters the state as a^(n-1-j) phi(k_j) v_j^T: phi(K) rows are
//   weighted a^(n-1-j), so the state update and z keep their MMAs;
//   P_rj then carries a^(r+1) a^(n-1-j) and the mask keeps a^(r-j) of it
//   (times a^(-n));
//   the held state is multiplied by a^n before the chunk's update.
// A state-pass part's record is its sum decayed to the part's last token;
// segment s starts from sum_p a^(tok0_s - end_p) record_p.

// Weighted sum of state records p0 .. p1-1 (as sum_states_to_tmem): record p
// covers tokens up to part_end(p) - 1 and is weighted a^(tok0 - part_end(p)).
template <int D>
__device__ __forceinline__ void sum_states_decayed(const float* recs, long long stride, int p0, int p1,
                                                   uint32_t lane_addr, uint32_t col, int row, float log2a,
                                                   int tok0, int F, int seg_len, int sub_len) {
#pragma unroll 1
  for (int h = 0; h < D; h += 64) {
    float4 acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row >= 0) {
#pragma unroll 1
      for (int p = p0; p < p1; ++p) {
        const int sg = p / F, part = p % F;
        const int pend = min(sg * seg_len + (part + 1) * sub_len, (sg + 1) * seg_len);
        const float w = exp2f((float)(tok0 - pend) * log2a);
        const float4* src = reinterpret_cast<const float4*>(recs + p * stride + (long long)row * D + h);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float4 f = src[j];
          acc[j].x = fmaf(w, f.x, acc[j].x); acc[j].y = fmaf(w, f.y, acc[j].y);
          acc[j].z = fmaf(w, f.z, acc[j].z); acc[j].w = fmaf(w, f.w, acc[j].w);
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

// The bf16 copy of the held state (as copy_state_to_smem) and, in the same
// pass, the held state multiplied by `f` in tensor memory (every lane).
template <int D>
__device__ __forceinline__ void copy_state_and_scale(uint32_t taddr, uint8_t* sbuf, int row, float f) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(taddr + c0, v);
    tmem_ld_wait();
    if (row >= 0) {
      const int b = c0 / 64, cb = (c0 % 64) / 8;
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
    uint32_t lo[16], hi[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      lo[j] = __float_as_uint(__uint_as_float(v[j]) * f);
      hi[j] = __float_as_uint(__uint_as_float(v[16 + j]) * f);
    }
    tmem_st16(taddr + c0, lo);
    tmem_st16(taddr + c0 + 16, hi);
  }
  tmem_st_wait();
}

// phi in place on a [C][D] tile in packed bf16 (as phi_tile_bf16), row r
// multiplied by a^(r+1) = 2^((r+1) log2a).
template <int D, int NT>
__device__ __forceinline__ void phi_tile_bf16_decayed(uint8_t* tile, int t, float log2a) {
  constexpr int PER = (C * D * 2 / 16) / NT;
#pragma unroll 1
  for (int i = 0; i < PER; ++i) {
    const int idx = t + NT * i;
    const int r = (idx & 1023) >> 3;                // 8 chunks of 16 bytes per 128-byte row
    const float w = exp2f((float)(r + 1) * log2a);
    const uint32_t w2 = pack_bf16x2(w, w);
    uint4 x = reinterpret_cast<const uint4*>(tile)[idx];
    uint32_t* px = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t f = phi_bf16x2(px[h]);
      asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(px[h]) : "r"(f), "r"(w2));
    }
    reinterpret_cast<uint4*>(tile)[idx] = x;
  }
}

template <int D, bool kDecay = false>
__global__ void __launch_bounds__(448, 1)
tc_forward_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                  const __grid_constant__ CUtensorMap map_o32, const FwdParams prm) {
  using G = Cfg<D>;
  using L = FwdSmem<D>;
  constexpr int ST = G::ST, NPB = G::NPB, NOB = G::NOB;
  static_assert(!kDecay || G::MERGE, "decay gating is laid out for D = 64");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  float* zst = reinterpret_cast<float*>(sm + L::OFF_ZST);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* full = bars;                          // [ST]
  uint64_t* phi_done = bars + ST;                 // [ST]
  uint64_t* empty = bars + 2 * ST;                // [ST]
  uint64_t* p_full = bars + 3 * ST;               // [NPB]
  uint64_t* p_ready = p_full + NPB;               // [NPB]
  uint64_t* o_full = p_ready + NPB;               // [NOB]
  uint64_t* o_empty = o_full + NOB;               // [NOB]
  uint64_t* s_full = o_empty + NOB;
  uint64_t* s_ready = s_full + 1;
  uint64_t* mma_fin = s_full + 2;
  uint64_t* ost_full = s_full + 3;                // [ST] output tile of the staged chunk written (group B)
  uint64_t* never = ost_full + ST;                // completed by nobody (timeout test)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::OFF_MISC + 4);
  // the swizzled operand boxes need 1024-byte alignment of the shared window
  // a backward launched after this forward (reading its records) may start
  // filling its pipeline as this grid's CTAs retire; it reads nothing this
  // kernel writes before its own dependency wait
  griddep_launch_dependents();
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(prm.status);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long rstride = rec_words<D>();
  int bh, tok0, tok_end, nchunks, nrec;
  bool last_seg;
  const float* recs;
  ChunkMap cmap;
  if (!kDecay && prm.NP > 0) {
    // piece blockIdx.x; its first head starts from the records of the
    // pieces before it in that head (one each), a later head from zero
    const long long g0 = (long long)blockIdx.x * prm.piece_len;
    const long long g1 = min((long long)prm.BH * prm.nch, g0 + prm.piece_len);
    bh = (int)(g0 / prm.nch);
    tok0 = (int)(g0 % prm.nch) * C;
    tok_end = prm.N;
    nchunks = (int)(g1 - g0);
    const long long first = (long long)bh * prm.nch / prm.piece_len;   // piece holding the head's start
    recs = prm.ws_state + first * rstride;
    nrec = (int)(blockIdx.x - first);
    last_seg = false;
    cmap = ChunkMap{g0, prm.nch, bh, tok0, prm.N, true};
  } else {
    // segment-major order: the first segments (which wait for no records) come first
    const int BH = gridDim.x / prm.P;
    bh = blockIdx.x % BH;
    const int seg = blockIdx.x / BH;
    tok0 = seg * prm.seg_len;
    tok_end = min(prm.N, tok0 + prm.seg_len);
    nchunks = (tok_end - tok0 + C - 1) / C;
    recs = prm.ws_state + (long long)bh * prm.P * prm.F * rstride;
    nrec = seg * prm.F;                   // records of the earlier segments
    last_seg = seg == prm.P - 1;
    cmap = ChunkMap{0, 0, bh, tok0, prm.N, false};
  }
  const float log2a = kDecay ? log2f(prm.alpha[bh % prm.H]) : 0.f;
  const bool write_final = last_seg && prm.S_final != nullptr;
  // the state update after the last chunk is only needed for the final state
  const int nupdates = write_final ? nchunks : nchunks - 1;

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
    for (int i = 0; i < NOB; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 128);
    }
    mbar_init(s_full, 1);
    mbar_init(s_ready, 128);
    mbar_init(mma_fin, 1);
    for (int i = 0; i < ST; ++i) mbar_init(&ost_full[i], 128);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (G::MERGE) {
    uint4* ones = reinterpret_cast<uint4*>(sm + L::OFF_ONES);
    for (int i = tid; i < BOX / 16; i += blockDim.x) ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
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
      if (!G::MERGE) tma_prefetch_desc(&map_o);
      // The output tile of a chunk is staged in its stage's Q region (dead
      // once the chunk's MMAs are done); this thread stores it with TMA and
      // waits until the store has read it before refilling the stage.
      auto store_out = [&](int c) {
        const int s = c % ST;
        if (!mbar_wait(&ost_full[s], (c / ST) & 1, abort_flag, kTimeoutNs)) return false;
        uint8_t* stg = sm + s * G::STAGE;
#pragma unroll
        for (int b = 0; b < G::NB; ++b) tma_store_3d(&map_o, stg + b * BOX, 64 * b, cmap.y_of(c), cmap.bh_of(c));
        tma_store_commit();
        tma_store_wait_read<0>();
        return true;
      };
      int issued = 0, stored = 0;
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST;
        if (c >= ST) {
          ok = mbar_wait(&empty[s], ((c / ST) - 1) & 1, abort_flag, kTimeoutNs);
          if (!ok) break;
        }
        uint8_t* stg = sm + s * G::STAGE;
        const int y = cmap.y_of(c), cbh = cmap.bh_of(c);
        mbar_arrive_expect_tx(&full[s], 3 * G::TILE);
        // K and V regions are free once the stage's MMAs are done; !MERGE:
        // the Q region holds the previous chunk's output until its store has
        // read it, so its load goes last
#pragma unroll
        for (int b = 0; b < G::NB; ++b) {
          tma_load_3d(stg + G::OFF_K + b * BOX, &map_k, &full[s], 64 * b, y, cbh);
          tma_load_3d(stg + G::OFF_V + b * BOX, &map_v, &full[s], 64 * b, y, cbh);
        }
        if (c >= ST && !G::MERGE) {
          ok = store_out(c - ST);
          if (!ok) {
            // the K and V loads of this stage are in flight: let them land
            issued = c + 1;
            break;
          }
          stored = c - ST + 1;
        }
#pragma unroll
        for (int b = 0; b < G::NB; ++b) tma_load_3d(stg + b * BOX, &map_q, &full[s], 64 * b, y, cbh);
        issued = c + 1;
      }
      // the chunks still in the ring: their outputs
      if (!G::MERGE)
        for (int c = stored; c < issued && ok; ++c) ok = store_out(c);
      // every store must be complete, and every issued load must have landed,
      // before the CTA's shared memory is released
      tma_store_wait<0>();
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_drain(&full[c % ST], (c / ST) & 1, kTimeoutNs);
    }
  } else if (warp == 13) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_qk = make_idesc_bf16(128, G::NQK, false, false);  // [P | O | den] or P
      constexpr uint32_t id_qs = make_idesc_bf16(128, D, false, false);    // O = phiQ S_prev (!MERGE)
      // S^T += V^T phiK; MERGE: [S^T ; z] += [V^T ; 1] phiK
      constexpr uint32_t id_vk = make_idesc_bf16(G::MERGE ? 128 : D, D, true, true);
      // O += P V; MERGE: [O | den] += P [V | 1]
      constexpr uint32_t id_pv = make_idesc_bf16(128, G::MERGE ? D + G::ZR : D, false, true);
      const uint32_t sbuf_a = smem_u32(sm + L::OFF_SBUF);
      const uint32_t ones_a = smem_u32(sm + L::OFF_ONES);
      // O += P V of chunk c once group B has packed its P; frees the stage
      auto issue_pv = [&](int c) -> bool {
        const int s = c % ST, pb = c % NPB, ob = c % NOB;
        const uint32_t va = smem_u32(sm + s * G::STAGE) + G::OFF_V;
        const uint64_t dv = make_sdesc(va, G::MERGE ? ones_a - va : (uint32_t)BOX, 1024, kSwizzle128B);
        if (!mbar_wait(&p_ready[pb], (c / NPB) & 1, abort_flag, kTimeoutNs)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ts(tmem + G::ocol(ob), tmem + G::pcol(pb) + k * 8, sdesc_add(dv, k * 2048), id_pv, 1);
        tc_commit(&o_full[ob]);
        tc_commit(&empty[s]);
        return true;
      };
      // timeout test: a wait that can only give up (no MMA is issued)
      bool ok = prm.timeout_test ? mbar_wait(never, 0, abort_flag, kTimeoutNs) : true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST;
        const uint32_t qa = smem_u32(sm + s * G::STAGE);
        const uint32_t ka = qa + G::OFF_K;
        const uint32_t va = qa + G::OFF_V;
        // the second 64-wide block of an MN-major V operand: the next feature
        // box, or (MERGE) the ones tile
        const uint32_t v_lbo = G::MERGE ? ones_a - va : (uint32_t)BOX;
        const int pb = c % NPB, ob = c % NOB;
        const uint32_t pc = tmem + G::pcol(pb), oc = tmem + G::ocol(ob);
        ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        // O buffer ob is free once the epilogue of chunk c - NOB has read it
        if (ok && G::MERGE && c >= NOB) ok = mbar_wait(&o_empty[ob], ((c / NOB) - 1) & 1, abort_flag, kTimeoutNs);
        if (ok && G::MERGE) ok = mbar_wait(s_ready, c & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        // operand descriptors of this stage; each k-step adds a constant
        const uint64_t dq = make_sdesc(qa, 16, 1024, kSwizzle128B);
        const uint64_t dk = make_sdesc(ka, 16, 1024, kSwizzle128B);
        // V (MN-major, second 64-wide block at v_lbo) and phi(K) (MN-major)
        const uint64_t dv = make_sdesc(va, v_lbo, 1024, kSwizzle128B);
        const uint64_t dkm = make_sdesc(ka, BOX, 1024, kSwizzle128B);
        auto issue_state = [&]() -> bool {
#pragma unroll
          for (int k = 0; k < C / 16; ++k)
            mma_ss(tmem + G::COL_S, sdesc_add(dv, k * 2048), sdesc_add(dkm, k * 2048), id_vk, 1);
          tc_commit(s_full);
          return true;
        };
        // P (and with MERGE, O = phiQ S_prev in the next D columns)
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * BOX + (k & 3) * 32;
          mma_ss(pc, sdesc_add(dq, off), sdesc_add(dk, off), id_qk, k > 0);
        }
        tc_commit(&p_full[pb]);
        if (!G::MERGE) {
          ok = mbar_wait(s_ready, c & 1, abort_flag, kTimeoutNs);
          if (ok && c >= NOB) ok = mbar_wait(&o_empty[ob], ((c / NOB) - 1) & 1, abort_flag, kTimeoutNs);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ds = make_sdesc(sbuf_a, 16, 1024, kSwizzle128B);
#pragma unroll
          for (int k = 0; k < G::KSTEPS; ++k)
            mma_ss(oc, sdesc_add(dq, (k >> 2) * BOX + (k & 3) * 32), sdesc_add(ds, (k >> 2) * (D * 128) + (k & 3) * 32),
                   id_qs, k > 0);
        }
        // MERGE: P V lags one chunk and goes before this chunk's state
        // update, so the tensor pipe runs it while group B packs P of this
        // chunk, and its O buffer is released early.
        // !MERGE: the state copy buffer is shared by all stages and may be
        // refilled once s_full shows that every earlier MMA is done, so the
        // update comes after this chunk's O MMA.
        if (G::MERGE) {
          if (c > 0) ok = issue_pv(c - 1);
          if (ok && c < nupdates) ok = issue_state();
        } else {
          if (c < nupdates) ok = issue_state();
          if (ok) ok = issue_pv(c);
        }
      }
      if (G::MERGE && ok && nchunks > 0) ok = issue_pv(nchunks - 1);
      // every MMA issued must have finished before tensor memory is released
      tc_commit(mma_fin);
      mbar_drain(mma_fin, 0, kTimeoutNs);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- group A: phi(Q), state copy ----------------
    const int t = tid - 128;                // 0..127
    const int q = warp & 3;                 // TMEM quadrant of this warp
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    // this lane's row of the held state: value index m of S^T (row < 0: none).
    // MERGE (M = 128 layout): lanes 0..D-1 hold S^T; lanes D.. hold z, whose
    // record slice starts right after the D x D part (row D); the copy takes
    // ZR of them as its rows D..D+ZR-1
    const int row = G::MERGE ? (q < 2 ? 32 * q + lane : -1) : state_row<D>(q, lane);
    const int row_sum = G::MERGE && q >= 2 ? D : row;
    const int row_copy = G::MERGE && q == 2 ? (lane < G::ZR ? D + lane : -1) : row;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      if constexpr (kDecay)
        phi_tile_bf16_decayed<D, 128>(sm + s * G::STAGE, t, log2a);   // Q, row r times a^(r+1)
      else
        phi_tile_bf16<D, 128>(sm + s * G::STAGE, t);   // Q
      fence_proxy_async_smem();
      mbar_arrive(&phi_done[s]);
      if (c == 0) {
        // this segment's starting state: the sum of the earlier segments' records
        if (nrec > 0) griddep_wait();
        if constexpr (kDecay)
          sum_states_decayed<D>(recs, rstride, 0, nrec, lane_addr, G::COL_S, row_sum, log2a, tok0, prm.F,
                                prm.seg_len, prm.sub_len);
        else if constexpr (G::MERGE)
          // centred records: S^T rows add the sum of their value component,
          // the z rows the token count tok0
          sum_states_to_tmem<D>(recs, rstride, 0, nrec, lane_addr, G::COL_S, row_sum,
                                centred_row_add<D>(recs, rstride, 0, nrec, row_sum, (float)tok0));
        else
          sum_states_to_tmem<D>(recs, rstride, 0, nrec, lane_addr, G::COL_S, row_sum);
      } else {
        // the state after chunk c - 1's update
        ok = mbar_wait(s_full, (c - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        // a piece's next head starts from zero (a sum of no records)
        if (!kDecay && !G::MERGE && cmap.head_start(c))
          sum_states_to_tmem<D>(recs, rstride, 0, 0, lane_addr, G::COL_S, row_sum);
      }
      if constexpr (kDecay) {
        // the copy of S_prev, and the held state decayed by a^n before this
        // chunk's n tokens are added
        const int n_valid = min(C, tok_end - (tok0 + c * C));
        copy_state_and_scale<D>(lane_addr + G::COL_S, sm + s * G::STAGE + G::OFF_SB, row_copy,
                                exp2f((float)n_valid * log2a));
      } else {
        copy_state_to_smem<D>(lane_addr + G::COL_S, G::MERGE ? sm + s * G::STAGE + G::OFF_SB : sm + L::OFF_SBUF,
                              row_copy);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(s_ready);
    }
    if (ok && write_final) {
      ok = mbar_wait(mma_fin, 0, abort_flag, kTimeoutNs);
      if (ok) {
        tc_fence_after();
        store_state_transposed<D>(prm.S_final + (long long)bh * D * D, lane_addr, G::COL_S, row);
        if (G::MERGE && kDecay && q == 2) {
          // z from the first z lane (without decay group C writes the exact sums)
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(lane_addr + G::COL_S + c0, v);
            tmem_ld_wait();
            if (lane == 0)
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(prm.z_final + (long long)bh * D + c0 + j) =
                    make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                __uint_as_float(v[j + 3]));
          }
        }
      }
    }
  } else if (warp >= 8 && warp < 12) {
    // ---------------- group B: P, denominators and the output epilogue ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;            // chunk row (query token) of this thread
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    // Masked P row of chunk c in bf16, packed into the first 64 columns of its
    // buffer (!MERGE: with its fp32 row sum; MERGE: P V sums the packed row).
    // Warp q holds rows 32q..32q+31: 32-column pieces left of q are kept
    // whole, piece q keeps columns <= lane, pieces right of q are zero.
    // Returns with the packed row written (tmem_st_wait) but not yet published.
    auto p_pass = [&](int c, float& rowsum) -> bool {
      const int s = c % ST, pb = c % NPB;
      const uint32_t pcol = G::pcol(pb);
      // (!MERGE: the phi(Q) tile is read afterwards for phi(q) . z_prev)
      if (!mbar_wait(&p_full[pb], (c / NPB) & 1, abort_flag, kTimeoutNs)) return false;
      if (!G::MERGE && !mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs)) return false;
      tc_fence_after();
      rowsum = 0.f;
      // with decay, the kept entries carry a^(r-j+n): times a^(-n)
      const float dfac = kDecay ? exp2f(-(float)min(C, tok_end - (tok0 + c * C)) * log2a) : 1.f;
#pragma unroll 1
      for (int p = 0; p < 4; ++p) {
        uint32_t pk[16];
        if (p < q) {
          uint32_t v[32];
          tmem_ld32(lane_addr + pcol + 32 * p, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float a = __uint_as_float(v[2 * j]), b = __uint_as_float(v[2 * j + 1]);
            if (kDecay) {
              a *= dfac;
              b *= dfac;
            }
            if (!G::MERGE) rowsum += a + b;
            pk[j] = pack_bf16x2(a, b);
          }
        } else if (p == q) {
          uint32_t v[32];
          tmem_ld32(lane_addr + pcol + 32 * p, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a = (2 * j <= lane) ? __uint_as_float(v[2 * j]) * dfac : 0.f;
            const float b = (2 * j + 1 <= lane) ? __uint_as_float(v[2 * j + 1]) * dfac : 0.f;
            if (!G::MERGE) rowsum += a + b;
            pk[j] = pack_bf16x2(a, b);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = 0u;
        }
        tmem_st16(lane_addr + pcol + 16 * p, pk);
      }
      tmem_st_wait();
      return true;
    };
    // Output rows of chunk c, scaled by inv_den (MERGE: read from the den
    // column here), staged as swizzled bf16 rows. !MERGE: in the chunk's Q
    // tile region; the TMA producer stores the whole tile (rows past the end
    // of the sequence are clipped) before it refills the stage. MERGE: in
    // output tile c % 2; this warp stores its 32 rows itself once the store of
    // chunk c - 2 has finished reading the tile.
    auto epilogue = [&](int c, float inv_den) -> bool {
      const int s = c % ST, ob = c % NOB;
      const uint32_t ocol = G::ocol(ob);
      if (!mbar_wait(&o_full[ob], (c / NOB) & 1, abort_flag, kTimeoutNs)) return false;
      tc_fence_after();
      uint8_t* ost = G::MERGE ? sm + L::OFF_OUT + ob * G::TILE : sm + s * G::STAGE;
      // scale, pack and stage 32 columns of the row
      auto put32 = [&](int c0, const uint32_t (&v)[32]) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * inv_den, __uint_as_float(v[8 * j + 1]) * inv_den);
          w.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv_den, __uint_as_float(v[8 * j + 3]) * inv_den);
          w.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv_den, __uint_as_float(v[8 * j + 5]) * inv_den);
          w.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv_den, __uint_as_float(v[8 * j + 7]) * inv_den);
          *reinterpret_cast<uint4*>(ost + (c0 / 64) * BOX + sw128(r, (c0 % 64) / 8 + j)) = w;
        }
      };
      if constexpr (G::MERGE) {
        // the whole row and den = phi(q_r) . z_prev + the row sum of the
        // packed P row, read at once, so the O buffer is released early
        uint32_t v0[32], v1[32], dw;
        tmem_ld32(lane_addr + ocol, v0);
        tmem_ld32(lane_addr + ocol + 32, v1);
        tmem_ld1(lane_addr + ocol + D, dw);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&o_empty[ob]);
        inv_den = 1.f / (__uint_as_float(dw) + prm.eps);
        if (c >= 2) {
          if (lane == 0) tma_store_wait_read<1>();
          __syncwarp();
        }
        put32(0, v0);
        put32(32, v1);
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(lane_addr + ocol + c0, v);
          tmem_ld_wait();
          put32(c0, v);
        }
        tc_fence_before();
        mbar_arrive(&o_empty[ob]);
      }
      fence_proxy_async_smem();
      if constexpr (G::MERGE) {
        __syncwarp();
        if (lane == 0) {
          // one bulk group per chunk (empty past the end of the sequence), so
          // that waiting for all but the newest group frees tile ob
          const int y = tok0 + c * C + 32 * q;
          if (y < prm.N) tma_store_3d(&map_o32, ost + 32 * q * 128, 0, y, bh);
          tma_store_commit();
        }
      } else {
        mbar_arrive(&ost_full[s]);
      }
      return true;
    };
    bool ok = true;
    if constexpr (G::MERGE) {
      // P V of chunk c is issued after the MMAs of chunk c + 1, so the P pass
      // of chunk c + 1 comes before the epilogue of chunk c
      for (int c = 0; c <= nchunks && ok; ++c) {
        if (c < nchunks) {
          float unused;
          ok = p_pass(c, unused);
          if (!ok) break;
          tc_fence_before();
          mbar_arrive(&p_ready[c % NPB]);
        }
        if (c >= 1) ok = epilogue(c - 1, 0.f);
      }
    } else {
      for (int c = 0; c < nchunks && ok; ++c) {
        float rowsum;
        ok = p_pass(c, rowsum);
        if (!ok) break;
        // phi(q_r) . z_prev from the phi-transformed Q tile (swizzled rows)
        float dot = 0.f;
        {
          const int s = c % ST;
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
        tc_fence_before();
        mbar_arrive(&p_ready[c % NPB]);
        ok = epilogue(c, 1.f / (rowsum + dot + prm.eps));
      }
    }
    // every store must be complete before the CTA's shared memory is released
    if (G::MERGE && lane == 0) tma_store_wait<0>();
  } else {
    // ---------------- group C: phi(K) and (!MERGE) z ----------------
    using X = ExactLayout<D, 128>;
    const int t = tid;                      // 0..127
    const int fc = X::FCW * (t >> 5) + (lane % X::FCW);
    const bool owner = lane < X::FCW;       // holds the z of features 8 fc .. 8 fc + 7
    float zrun[8];
    // MERGE without decay, last segment with a final state: per-thread
    // partial sums of the exact fp32 phi(k) for the exported z
    float zfin[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) zfin[e] = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      const int n_valid = kDecay ? min(C, tok_end - (tok0 + c * C)) : cmap.n_valid(c);
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      float colsum[8];
      if constexpr (G::MERGE) {
        // z is summed by the state MMA; with decay, row j is weighted a^(n-1-j)
        if constexpr (kDecay)
          phi_tile_exact<D, 128, false, false, true>(sm + s * G::STAGE + G::OFF_K, t, n_valid, colsum, log2a,
                                                     n_valid - 1);
        else if (write_final)
          phi_tile_exact<D, 128, false, true>(sm + s * G::STAGE + G::OFF_K, t, n_valid, zfin);  // K, sums
        else
          phi_tile_exact<D, 128, false, false>(sm + s * G::STAGE + G::OFF_K, t, n_valid, colsum);  // K
        fence_proxy_async_smem();
        mbar_arrive(&phi_done[s]);
        continue;
      }
      phi_tile_exact<D, 128>(sm + s * G::STAGE + G::OFF_K, t, n_valid, colsum);  // K
      fence_proxy_async_smem();
      if (c == 0) {
        if (nrec > 0) griddep_wait();
        sum_vectors8<D>(recs, rstride, 0, nrec, 8 * fc, zrun);
      } else if (cmap.head_start(c)) {
#pragma unroll
        for (int e = 0; e < 8; ++e) zrun[e] = 0.f;
      }
      if (owner) {
        // z before this chunk, for group B's denominators
        float4* zd = reinterpret_cast<float4*>(zst + s * D + 8 * fc);
        zd[0] = make_float4(zrun[0], zrun[1], zrun[2], zrun[3]);
        zd[1] = make_float4(zrun[4], zrun[5], zrun[6], zrun[7]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) zrun[e] += colsum[e];
      mbar_arrive(&phi_done[s]);
    }
    if (G::MERGE && !kDecay && ok && write_final) {
      // z = (sum of the centred records' z_psi) + tok0 + this segment's exact sums
      reduce_row_groups<D, 128>(zfin);
      if (nrec > 0) griddep_wait();
      sum_vectors8<D>(recs, rstride, 0, nrec, 8 * fc, zrun);
#pragma unroll
      for (int e = 0; e < 8; ++e) zrun[e] += (float)tok0 + zfin[e];
    }
    if ((!G::MERGE || !kDecay) && ok && write_final && owner) {
      float4* zd = reinterpret_cast<float4*>(prm.z_final + (long long)bh * D + 8 * fc);
      zd[0] = make_float4(zrun[0], zrun[1], zrun[2], zrun[3]);
      zd[1] = make_float4(zrun[4], zrun[5], zrun[6], zrun[7]);
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
// Per-segment state sums: dS^T = V_seg^T phi(K_seg) on the tensor cores into
// TMEM (fp32), dz = column sums of phi(K_seg) on the CUDA cores (fp32), for
// segments 0 .. P-2 of each sequence (the last segment's sum is never read:
// the forward kernel's last segment carries the state to its end itself).
// 320 threads: warps 0-7 phi(K) (rounded to nearest) and z, warps 0-3 also
// the final store of dS^T; warp 8 TMA, warp 9 TMEM allocator and MMA.
// ---------------------------------------------------------------------------
template <int D>
struct StateSmem {
  // D = 64: the state MMA runs with M = 128, A = [V^T ; 1] (ones tile as the
  // second 64-wide block of A), so lanes 64.. of the accumulator hold dz
  static constexpr bool ZMMA = D == 64;
  static constexpr int OFF_ONES = Cfg<D>::ST_S * Cfg<D>::STAGE_S;
  static constexpr int OFF_BAR = OFF_ONES + (ZMMA ? BOX : 0);
  static constexpr int NBAR = 3 * Cfg<D>::ST_S + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
};

struct StateParams {
  int N, P, seg_len, F, sub_len;
  int nseg;         // segments summed: P - 1 (causal) or P (non-causal)
  float* ws_state;  // [BH][P*F][rec_words]
  int* status;
  const float* alpha = nullptr;   // kDecay: [H] per-head factors
  int H = 1;
  // balanced pieces (SegPlan): CTA i sums the part of piece i in its last
  // head into record i, if that head goes on after the piece
  int NP = 0, piece_len = 0, nch = 0, BH = 0;
};

// kDecay: each record is decayed to its part's last token (row j of a chunk
// weighted a^(part_end - 1 - token)).
// D = 64 without decay: centred records (see rec_words). The K tile becomes
// psi(K) = phi(K) - 1, the MMA is [S_psi^T | sum v ; . | .] = [V^T ; 1]
// [psi(K) | 1] (N = D + 16, the ones tile as the second 64-wide block of B,
// so accumulator column D of lane m is the sum of v_m), and z_psi is summed
// from the exact fp32 psi on the CUDA cores.
template <int D, bool kDecay = false>
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
  // the dependent forward kernel may start filling its pipeline right away
  griddep_launch_dependents();
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(prm.status);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bh, tok0, tok_end;
  long long rec_index;
  if (prm.NP > 0) {
    const long long g0 = (long long)blockIdx.x * prm.piece_len;
    const long long g1 = min((long long)prm.BH * prm.nch, g0 + prm.piece_len);
    const long long h = (g1 - 1) / prm.nch;
    if (g1 == (h + 1) * prm.nch) return;   // the piece ends its head: no record
    const long long s0 = max(g0, h * prm.nch);
    bh = (int)h;
    tok0 = (int)(s0 - h * prm.nch) * C;
    tok_end = min(prm.N, (int)(g1 - h * prm.nch) * C);
    rec_index = blockIdx.x;
  } else {
    // part j of segment j / F covers sub_len tokens from j % F * sub_len
    const int nparts = prm.nseg * prm.F;
    const int j = blockIdx.x % nparts;
    bh = blockIdx.x / nparts;
    const int seg = j / prm.F, part = j % prm.F;
    const int seg_end = min(prm.N, (seg + 1) * prm.seg_len);
    tok0 = seg * prm.seg_len + part * prm.sub_len;
    tok_end = min(seg_end, tok0 + prm.sub_len);
    rec_index = (long long)bh * prm.P * prm.F + j;
  }
  // a part past the end of a short last segment (non-causal) holds no token
  const int nchunks = max(0, (tok_end - tok0 + C - 1) / C);
  static_assert(!kDecay || StateSmem<D>::ZMMA, "decay gating is laid out for D = 64");
  constexpr bool kCentre = L::ZMMA && !kDecay;
  const float log2a = kDecay ? log2f(prm.alpha[bh % prm.H]) : 0.f;

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
  if constexpr (L::ZMMA) {
    uint4* ones = reinterpret_cast<uint4*>(sm + L::OFF_ONES);
    for (int i = tid; i < BOX / 16; i += blockDim.x) ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
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
        mbar_drain(&full[c % ST], (c / ST) & 1, kTimeoutNs);
    }
  } else if (warp == 9) {
    if (lane == 0) {
      // S^T += V^T phi(K); ZMMA: [S^T ; z] += [V^T ; 1] phi(K); kCentre:
      // [S_psi^T | sum v ; z_psi | n] += [V^T ; 1] [psi(K) | 1]
      constexpr uint32_t id_vk = make_idesc_bf16(L::ZMMA ? 128 : D, kCentre ? D + 16 : D, true, true);
      const uint32_t ones_a = smem_u32(sm + L::OFF_ONES);
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % ST;
        const uint32_t ka = smem_u32(sm + s * G::STAGE_S);
        const uint32_t va = ka + G::TILE;
        const uint64_t dv = make_sdesc(va, L::ZMMA ? ones_a - va : (uint32_t)BOX, 1024, kSwizzle128B);
        const uint64_t dk = make_sdesc(ka, kCentre ? ones_a - ka : (uint32_t)BOX, 1024, kSwizzle128B);
        ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          mma_ss(tmem, sdesc_add(dv, k * 2048), sdesc_add(dk, k * 2048), id_vk, (c > 0 || k > 0) ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      tc_commit(s_full);
      tc_commit(mma_fin);
      mbar_drain(mma_fin, 0, kTimeoutNs);
    }
  } else {
    using X = ExactLayout<D, 256>;
    const int t = tid;                      // 0..255
    const int q = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    // row of S^T held by this lane (ZMMA: M = 128 layout, lanes 0..D-1)
    const int row = L::ZMMA ? (q < 2 ? 32 * q + lane : -1) : state_row<D>(q, lane);
    const int fc = X::FCW * (t >> 5) + (lane % X::FCW);
    // per-thread partial column sums, reduced once after the last chunk
    float zrun[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) zrun[e] = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      const int n_valid = min(C, tok_end - (tok0 + c * C));
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      if (kDecay)
        phi_tile_exact<D, 256, false, false, true>(sm + s * G::STAGE_S, t, n_valid, zrun, log2a,
                                                   tok_end - 1 - (tok0 + c * C));
      else if (kCentre)
        phi_tile_exact<D, 256, false, true, false, true>(sm + s * G::STAGE_S, t, n_valid, zrun);
      else if (L::ZMMA)
        phi_tile_exact<D, 256, false, false>(sm + s * G::STAGE_S, t, n_valid, zrun);
      else
        phi_tile_exact<D, 256, false>(sm + s * G::STAGE_S, t, n_valid, zrun);
      fence_proxy_async_smem();
      mbar_arrive(&phi_done[s]);
    }
    reduce_row_groups<D, 256>(zrun);
    float* dst = prm.ws_state + rec_index * rec_words<D>();
    if ((!L::ZMMA || kCentre) && ok && lane < X::FCW) {
      float4* zd = reinterpret_cast<float4*>(dst + D * D + 8 * fc);
      zd[0] = make_float4(zrun[0], zrun[1], zrun[2], zrun[3]);
      zd[1] = make_float4(zrun[4], zrun[5], zrun[6], zrun[7]);
    }
    if (ok && warp < 4) ok = mbar_wait(s_full, 0, abort_flag, kTimeoutNs);
    if (ok && warp < 4) {
      tc_fence_after();
      if (nchunks > 0) {
        store_state_from_tmem<D>(dst, lane_addr, 0, row);
        if (kCentre) {
          // sum v_m from accumulator column D of lane m
          uint32_t vs;
          tmem_ld1(lane_addr + D, vs);
          tmem_ld_wait();
          if (row >= 0) dst[D * D + D + row] = __uint_as_float(vs);
        }
        if (L::ZMMA && !kCentre && q == 2) {
          // dz from the first z lane
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(lane_addr + c0, v);
            tmem_ld_wait();
            if (lane == 0)
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(dst + D * D + c0 + e) =
                    make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                __uint_as_float(v[e + 3]));
          }
        }
      } else {
        // no MMA wrote the accumulator: the empty part's record is zero
        // (its z entries were written from zrun = 0 unless ZMMA without kCentre)
        for (int i = t; i < (L::ZMMA && !kCentre ? D * D + D : D * D); i += 128) dst[i] = 0.f;
        if (kCentre)
          for (int i = t; i < D; i += 128) dst[D * D + D + i] = 0.f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // after the barrier: a warp that gave up late is seen too
  if (*abort_flag && tid == 0) report_timeout(prm.status);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS_S);
  }
}

// ---------------------------------------------------------------------------
// Non-causal output: every query reads the whole sequence's state
// ([LA-state] fig. 2, [LA-order]: the summary S_N = phi(K)^T V, z_N):
//   out = phi(Q_c) S_N / (phi(Q_c) z_N + eps)
// S_N^T and z_N are the sums of all segments' records. Per chunk one MMA group:
// phi(Q) times the bf16 copy of S_N^T, which at D = 64 also carries z_N as
// hi + lo rows so that the normaliser comes out of the same MMA (at D = 128 it
// is summed on the CUDA cores); the output is staged in the chunk's Q tile and
// stored with TMA.
// 320 threads: warps 0-3 group A (phi(Q); the state sum and its copy), warps
// 4-7 group B (den, epilogue), warp 8 TMA producer, warp 9 TMEM and MMA.
// ---------------------------------------------------------------------------
template <int D>
struct NcSmem {
  static constexpr int NB = D / 64;
  static constexpr int TILE = NB * BOX;
  static constexpr int ST = D == 64 ? 10 : 4;                      // Q tiles in flight (a stage holds its output until stored)
  // D = 64: z_N rides in the MMA as bf16 hi + lo rows D, D + 1 of the S_N^T
  // operand (rows D + 2 .. D + 15 zero), so one MMA with N = D + 16 gives
  // [O | phi(Q) z_hi | phi(Q) z_lo] (about 16 bits of z in the denominator)
  static constexpr bool ZMMA = D == 64;
  static constexpr int NO = ZMMA ? D + 16 : D;                     // MMA N and O buffer width
  static constexpr int SBUF = ZMMA ? NO * 128 : NB * D * 128;      // bf16 [S_N^T ; z rows], K-major
  static constexpr int OFF_SBUF = ST * TILE;
  static constexpr int OFF_Z = OFF_SBUF + SBUF;                    // [D] z_N
  static constexpr int OFF_BAR = OFF_Z + D * 4;
  static constexpr int NBAR = 3 * ST + 4 + 2;                      // full, phi_done, ost_full; o_full/o_empty [2]; s_ready, mma_fin
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
  static constexpr uint32_t COL_O = 0;                             // 2 x NO
  static constexpr uint32_t COL_S = 2 * NO;                        // D
  static constexpr uint32_t TMEM_COLS = D == 64 ? 256 : 512;
};

template <int D>
__global__ void __launch_bounds__(320, 1)
tc_noncausal_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_o,
                    const FwdParams prm) {
  using L = NcSmem<D>;
  constexpr int ST = L::ST;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sbuf = sm + L::OFF_SBUF;
  float* zn = reinterpret_cast<float*>(sm + L::OFF_Z);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* full = bars;                  // [ST]
  uint64_t* phi_done = bars + ST;         // [ST]
  uint64_t* ost_full = bars + 2 * ST;     // [ST]
  uint64_t* o_full = bars + 3 * ST;       // [2]
  uint64_t* o_empty = o_full + 2;         // [2]
  uint64_t* s_ready = o_full + 4;
  uint64_t* mma_fin = o_full + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::OFF_MISC + 4);
  // as in the causal chunk loop: a following backward may start early
  griddep_launch_dependents();
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(prm.status);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = gridDim.x / prm.P;
  const int bh = blockIdx.x % BH, seg = blockIdx.x / BH;
  const int tok0 = seg * prm.seg_len;
  const int tok_end = min(prm.N, tok0 + prm.seg_len);
  const int nchunks = (tok_end - tok0 + C - 1) / C;
  const long long rstride = rec_words<D>();
  const float* recs = prm.ws_state + (long long)bh * prm.P * prm.F * rstride;
  const int nrec = prm.P * prm.F;

  if (tid == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&phi_done[i], 128);
      mbar_init(&ost_full[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 128);
    }
    mbar_init(s_ready, 128);
    mbar_init(mma_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer; stores each chunk's output from its Q tile ----------------
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_o);
      auto store_out = [&](int c) {
        const int s = c % ST;
        if (!mbar_wait(&ost_full[s], (c / ST) & 1, abort_flag, kTimeoutNs)) return false;
#pragma unroll
        for (int b = 0; b < L::NB; ++b) tma_store_3d(&map_o, sm + s * L::TILE + b * BOX, 64 * b, tok0 + c * C, bh);
        tma_store_commit();
        tma_store_wait_read<0>();
        return true;
      };
      int issued = 0, stored = 0;
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST;
        if (c >= ST) {
          ok = store_out(c - ST);
          if (!ok) break;
          stored = c - ST + 1;
        }
        mbar_arrive_expect_tx(&full[s], L::TILE);
#pragma unroll
        for (int b = 0; b < L::NB; ++b) tma_load_3d(sm + s * L::TILE + b * BOX, &map_q, &full[s], 64 * b, tok0 + c * C, bh);
        issued = c + 1;
      }
      for (int c = stored; c < issued && ok; ++c) ok = store_out(c);
      tma_store_wait<0>();
      for (int c = max(0, issued - ST); c < issued; ++c)
        mbar_drain(&full[c % ST], (c / ST) & 1, kTimeoutNs);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer: O = phi(Q) S_N ----------------
    if (lane == 0) {
      constexpr uint32_t id_qs = make_idesc_bf16(128, L::NO, false, false);
      const uint32_t sb = smem_u32(sbuf);
      bool ok = mbar_wait(s_ready, 0, abort_flag, kTimeoutNs);
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % ST, ob = c & 1;
        ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs);
        if (ok && c >= 2) ok = mbar_wait(&o_empty[ob], ((c >> 1) - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qa = smem_u32(sm + s * L::TILE);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + L::COL_O + L::NO * ob, make_sdesc(qa + (k >> 2) * BOX + (k & 3) * 32, 16, 1024, kSwizzle128B),
                 make_sdesc(sb + (k >> 2) * (D * 128) + (k & 3) * 32, 16, 1024, kSwizzle128B), id_qs, k > 0);
        tc_commit(&o_full[ob]);
      }
      tc_commit(mma_fin);
      mbar_drain(mma_fin, 0, kTimeoutNs);
    }
  } else if (warp < 4) {
    // ---------------- group A: S_N, z_N; phi(Q) ----------------
    const int t = tid;                      // 0..127
    const int q = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    const int row = state_row<D>(q, lane);
    griddep_wait();
    // D = 64: centred records (S^T rows add the sum of their value
    // component, z adds the token count N)
    sum_states_to_tmem<D>(recs, rstride, 0, nrec, lane_addr, L::COL_S, row,
                          L::ZMMA ? centred_row_add<D>(recs, rstride, 0, nrec, row, (float)prm.N) : 0.f);
    copy_state_to_smem<D>(lane_addr + L::COL_S, sbuf, row);
    for (int i = t; i < D; i += 128) {
      float acc = L::ZMMA ? (float)prm.N : 0.f;
      for (int p = 0; p < nrec; ++p) acc += recs[p * rstride + D * D + i];
      zn[i] = acc;
      if constexpr (L::ZMMA) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
        const __nv_bfloat16 lo = __float2bfloat16_rn(acc - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat16*>(sbuf + sw128(D, i >> 3) + 2 * (i & 7)) = hi;
        *reinterpret_cast<__nv_bfloat16*>(sbuf + sw128(D + 1, i >> 3) + 2 * (i & 7)) = lo;
      }
    }
    if constexpr (L::ZMMA)
      for (int i = t; i < (L::NO - D - 2) * 8; i += 128)
        *reinterpret_cast<uint4*>(sbuf + sw128(D + 2 + (i >> 3), i & 7)) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(s_ready);
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST;
      ok = mbar_wait(&full[s], (c / ST) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      phi_tile_bf16<D, 128>(sm + s * L::TILE, t);
      fence_proxy_async_smem();
      mbar_arrive(&phi_done[s]);
    }
    if (ok && seg == 0 && prm.S_final != nullptr) {
      // the final state (the same for every segment; written once per sequence)
      store_state_transposed<D>(prm.S_final + (long long)bh * D * D, lane_addr, L::COL_S, row);
      for (int i = t; i < D; i += 128) prm.z_final[(long long)bh * D + i] = zn[i];
    }
  } else {
    // ---------------- group B: den, epilogue ----------------
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
    bool ok = mbar_wait(s_ready, 0, abort_flag, kTimeoutNs);
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % ST, ob = c & 1;
      ok = mbar_wait(&phi_done[s], (c / ST) & 1, abort_flag, kTimeoutNs) &&
           mbar_wait(&o_full[ob], (c >> 1) & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      uint8_t* qt = sm + s * L::TILE;
      float dot = 0.f;
      if constexpr (L::ZMMA) {
        uint32_t dz[2];
        tmem_ld2(lane_addr + L::COL_O + L::NO * ob + D, dz);
        tmem_ld_wait();
        dot = __uint_as_float(dz[0]) + __uint_as_float(dz[1]);
      } else {
#pragma unroll 1
      for (int b = 0; b < L::NB; ++b)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 w = *reinterpret_cast<const uint4*>(qt + b * BOX + sw128(r, ch));
          const uint32_t* pw = reinterpret_cast<const uint32_t*>(&w);
          const float4 z0 = *reinterpret_cast<const float4*>(zn + b * 64 + ch * 8);
          const float4 z1 = *reinterpret_cast<const float4*>(zn + b * 64 + ch * 8 + 4);
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
      const float inv_den = 1.f / (dot + prm.eps);
      // the row of phi(Q) has been read: the Q tile takes the output row
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(lane_addr + L::COL_O + L::NO * ob + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * inv_den, __uint_as_float(v[8 * j + 1]) * inv_den);
          w.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv_den, __uint_as_float(v[8 * j + 3]) * inv_den);
          w.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv_den, __uint_as_float(v[8 * j + 5]) * inv_den);
          w.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv_den, __uint_as_float(v[8 * j + 7]) * inv_den);
          *reinterpret_cast<uint4*>(qt + (c0 / 64) * BOX + sw128(r, (c0 % 64) / 8 + j)) = w;
        }
      }
      tc_fence_before();
      mbar_arrive(&o_empty[ob]);
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
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool kDecay = false>
cudaError_t launch_state(const FwdArgs& a, const float* alpha = nullptr, int H = 1) {
  // causal: the segments before the last (none with one segment); non-causal:
  // all; with pieces, one CTA per piece (those that end their head exit)
  const int nseg = a.causal ? a.plan.P - 1 : a.plan.P;
  const bool pieces = !kDecay && a.plan.NP > 0;
  if (!pieces && nseg < 1) return cudaSuccess;
  CUtensorMap mk, mv;
  cudaError_t e = make_map(&mk, a.k, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mv, a.v, a.BH, a.N, D);
  if (e != cudaSuccess) return e;
  constexpr int smem = StateSmem<D>::BYTES;
  e = cudaFuncSetAttribute(tc_state_kernel<D, kDecay>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  StateParams p{a.N, a.plan.P, a.plan.seg_len, a.plan.F, state_sub_len(a.plan), nseg, a.ws_state,
                device_status_ptr()};
  p.alpha = alpha;
  p.H = H;
  if (pieces) {
    p.NP = a.plan.NP;
    p.piece_len = a.plan.piece_len;
    p.nch = (a.N + C - 1) / C;
    p.BH = a.BH;
  }
  const unsigned grid = pieces ? (unsigned)a.plan.NP : (unsigned)(a.BH * nseg * a.plan.F);
  tc_state_kernel<D, kDecay><<<grid, 320, smem, a.stream>>>(mk, mv, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <int D>
cudaError_t launch_noncausal(const FwdArgs& a) {
  CUtensorMap mq, mo;
  cudaError_t e = make_map(&mq, a.q, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mo, a.out, a.BH, a.N, D);
  if (e != cudaSuccess) return e;
  constexpr int smem = NcSmem<D>::BYTES;
  e = cudaFuncSetAttribute(tc_noncausal_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  FwdParams p{a.N, a.plan.P, a.plan.seg_len, a.plan.F, a.eps, a.ws_state, (__nv_bfloat16*)a.out,
              a.S_final, a.z_final, device_status_ptr()};
  // a dependent of the state kernel: its Q loads and phi(Q) overlap that
  // kernel; the state sum waits for the records
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.BH * a.plan.P);
  cfg.blockDim = dim3(320);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, tc_noncausal_kernel<D>, mq, mo, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <int D, bool kDecay = false>
cudaError_t launch_forward(const FwdArgs& a, const float* alpha = nullptr, int H = 1) {
  if (!kDecay && !a.causal) return launch_noncausal<D>(a);
  CUtensorMap mq, mk, mv, mo, mo32;
  cudaError_t e = make_map(&mq, a.q, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mk, a.k, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mv, a.v, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mo, a.out, a.BH, a.N, D);
  if (e == cudaSuccess) e = make_map(&mo32, a.out, a.BH, a.N, D, 32);
  if (e != cudaSuccess) return e;
  constexpr int smem = FwdSmem<D>::BYTES;
  e = cudaFuncSetAttribute(tc_forward_kernel<D, kDecay>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  FwdParams p{a.N, a.plan.P, a.plan.seg_len, a.plan.F, a.eps, a.ws_state, (__nv_bfloat16*)a.out,
              a.S_final, a.z_final, device_status_ptr()};
  p.alpha = alpha;
  p.H = H;
  p.sub_len = state_sub_len(a.plan);
  p.timeout_test = (!kDecay && take_timeout_test()) ? 1 : 0;
  const bool pieces = !kDecay && a.plan.NP > 0;
  if (pieces) {
    p.NP = a.plan.NP;
    p.piece_len = a.plan.piece_len;
    p.nch = (a.N + C - 1) / C;
    p.BH = a.BH;
  }
  // a dependent of the state kernel (when there is one): it may start before
  // that kernel ends and waits for its records only where it reads them
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(pieces ? a.plan.NP : a.BH * a.plan.P);
  cfg.blockDim = dim3(448);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.plan.P > 1 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, tc_forward_kernel<D, kDecay>, mq, mk, mv, mo, mo32, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace

bool tc_forward_supported(int dk, int dv, la_dtype dtype, int causal) {
  (void)causal;
  return dtype == LA_BF16 && dk == dv && (dk == 64 || dk == 128);
}

cudaError_t tc_forward_decay(const FwdArgs& a, const float* alpha, int H) {
  if (a.dk != 64 || a.dv != 64 || a.dtype != LA_BF16 || !a.causal) return cudaErrorInvalidValue;
  prof_begin(LA_SPAN_FWD_STATE, a.stream);
  cudaError_t e = launch_state<64, true>(a, alpha, H);
  prof_end(LA_SPAN_FWD_STATE, a.stream);
  if (e != cudaSuccess) return e;
  prof_begin(LA_SPAN_FWD_OUTPUT, a.stream);
  e = launch_forward<64, true>(a, alpha, H);
  prof_end(LA_SPAN_FWD_OUTPUT, a.stream);
  return e;
}

cudaError_t tc_segment_state(const FwdArgs& a) {
  return a.dk == 128 ? launch_state<128>(a) : launch_state<64>(a);
}

cudaError_t tc_forward_output(const FwdArgs& a) {
  return a.dk == 128 ? launch_forward<128>(a) : launch_forward<64>(a);
}

}  // namespace la
