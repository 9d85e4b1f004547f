// Multi-token decode on the tensor cores (bf16 tokens, dk = dv = 128, fp32
// state): T consecutive tokens of one (batch, head) per call, in groups of up
// to TG = 16, the state read and written once per call.
//
// The recurrence ("Linear Attention: KV를 고정 크기 상태에 누적하기", section
// "상태 갱신과 읽기를 식으로 정리하기") over a group of n tokens starting from
// S_0, z_0, in its chunked form (the masked sums of "상태공간모델·선형
// 어텐션", section 2, re-associated):
//   num_t = S_0^T phi(q_t) + sum_{j <= t} (phi(q_t) . phi(k_j)) v_j
//   den_t = phi(q_t) . z_0 + sum_{j <= t} phi(q_t) . phi(k_j) + eps
//   S    <- S_0 + sum_j phi(k_j) v_j^T,   z <- z_0 + sum_j phi(k_j)
// with phi(k) = 1 + psi(k) and psi = psi_hi + psi_lo (two bf16 parts, about
// 16 bits). The state is held transposed in tensor memory, S^T (lane = value
// index c, column = key index i), in fp32, with a bf16 copy of it beside.
// Per group two passes of MMAs (M = 128):
//   pass 1   D_P[t][.] = phi(q_t) [psi_hi ; z_hi ; z_lo ; 1]^T + phi(q_t) psi_lo^T
//            (N = 32: the scores against the group's keys without their 1,
//            phi(q_t) . z_0 and s_t = sum_i phi(q_t)_i; rows t >= 16 unused)
//            D[c][t] = S^T (bf16 copy) x phi(Q)^T                  (the read)
//   CUDA cores: P_tj = D_P[t][j] + s_t masked to j <= t < n, den_t
//   pass 2   D[c][t] += V^T P^T                                    (intra-group)
//            S^T += V^T 1 + V^T psi_hi + V^T psi_lo               (update)
// The update carries the common 1 of phi(k) exactly (V^T times a tile of
// ones) and psi to about 16 bits, so the state keeps fp32 accuracy; the read
// rounds the state and phi(q) to bf16, as the chunked forward does. z is
// updated in fp32 from 1 + psi_hi + psi_lo.
//
// Decay gating ("Linear Attention, 곱의 순서를 바꾸면 생기는 일", paragraph on
// 감쇠 게이팅; per-head factor a): S_t = a S_{t-1} + phi(k_t) v_t^T and z
// likewise, so over a group
//   num_t = a^(t+1) S_0^T phi(q_t) + sum_{j <= t} a^(t-j) (phi(q_t) . phi(k_j)) v_j
//   den_t = a^(t+1) phi(q_t) . z_0 + sum_{j <= t} a^(t-j) phi(q_t) . phi(k_j) + eps
//   S    <- a^n S_0 + sum_j a^(n-1-j) phi(k_j) v_j^T
// The read takes a second phi(Q) tile with row t weighted a^(t+1); the P
// pass keeps the unweighted one and the CUDA cores weight P_tj by a^(t-j)
// (and phi(q_t) . z_0 by a^(t+1)); the update's B tiles carry w_j =
// a^(n-1-j) as bf16 hi + lo rows (for the 1 of phi(k)) and w_j psi(k_j) as
// hi + lo, so the state keeps the accuracy of the undecayed update; the held
// state is multiplied by a^n in the pass that makes its bf16 copy.
//
// A persistent CTA per SM (a kernel that allocates tensor memory runs one
// CTA per SM) with two teams of 128 threads, each working through its own
// states with its own shared memory, half of tensor memory and its own
// barriers; team 1 starts half a state late, so that the two teams' memory
// phases alternate. Thread c of a team (warp c / 32 of it) owns lane c:
// value index c of the state and of the outputs, key index c of z. The state
// arrives as one 64 KB bulk copy into shared memory, from which thread c
// moves column c into tensor memory; the next state's copy then goes into
// the same buffer while this one runs. The updated state leaves from tensor
// memory straight to global memory (a warp writes 32 consecutive values of a
// row per store). Every wait is bounded; on a timeout the CTA stops and
// reports through the device status word.
#include <algorithm>

#include "la_tc_common.cuh"
#include "la_variants.cuh"

namespace la {

namespace {

using namespace sm100;

constexpr int DT = 128;                 // dk = dv
constexpr int TG = 16;                  // tokens per group
constexpr int TBOX = TG * 128;          // bytes of one [16 rows][64 bf16] SW128 box
constexpr int TTILE = 2 * TBOX;         // a [16][128] bf16 tile (two boxes)

constexpr int KROWS = 32;                // rows of the psi tiles (16 keys, then z_hi, z_lo, ones)
constexpr int KBOX = KROWS * 128;       // bytes of one [32 rows][64 bf16] SW128 box

template <bool kDecay>
struct DecTcT {
  static constexpr int OFF_SST = 0;                         // fp32 [128][128] state (bulk load)
  static constexpr int OFF_Q = OFF_SST + DT * DT * 4;       // phi(Q) bf16, K-major [t][i] (16 rows)
  static constexpr int OFF_KH = OFF_Q + TTILE;              // [psi_hi ; z_hi ; z_lo ; 1 ; 0] [32][128]
  static constexpr int OFF_KL = OFF_KH + 2 * KBOX;          // [psi_lo ; 0] [32][128]
  static constexpr int OFF_V = OFF_KL + 2 * KBOX;           // V bf16 [t][c] (16 rows)
  static constexpr int OFF_ONES = OFF_V + TTILE;            // ones [16][128]
  static constexpr int OFF_P = OFF_ONES + TTILE;            // P bf16, K-major [t][j] (j < 16 used)
  // decay: phi(Q) rows weighted a^(t+1) (the read), and the update's B tiles
  // [w_lo], [w psi]_hi, [w psi]_lo, each [16][128] ([w_hi] takes the place
  // of the ones tile, which the decayed update does not use)
  static constexpr int OFF_QS = OFF_P + TBOX;
  static constexpr int OFF_UW = OFF_QS + (kDecay ? TTILE : 0);
  static constexpr int OFF_Z = OFF_UW + (kDecay ? 3 * TTILE : 0);   // fp32 z [128]
  static constexpr int OFF_DEN = OFF_Z + DT * 4;            // fp32 1 / den [16]
  static constexpr int OFF_BAR = OFF_DEN + TG * 4;          // 3 mbarriers
  // one team's region, 1024-aligned; the CTA holds two, then the tensor-
  // memory slot and the abort flag
  static constexpr int TEAM_BYTES = (OFF_BAR + 24 + 1023) / 1024 * 1024;
  static constexpr int BYTES = 2 * TEAM_BYTES + 16;
  static_assert(OFF_Q % 1024 == 0 && OFF_KH % 1024 == 0 && OFF_KL % 1024 == 0 && OFF_V % 1024 == 0 &&
                    OFF_ONES % 1024 == 0 && OFF_P % 1024 == 0 && OFF_QS % 1024 == 0 && OFF_UW % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  // the P pass reads 128 rows of phi(Q) (rows 16.. are whatever follows in
  // shared memory; their results are never read): inside the team's region
  static_assert(OFF_Q + TBOX + 16 * 1024 <= TEAM_BYTES, "phi(Q) read as M = 128 stays in the region");
  static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
  // tensor memory columns (per team)
  static constexpr uint32_t COL_S = 0;                      // S^T fp32, 128 columns
  static constexpr uint32_t COL_SB = 128;                   // S^T bf16 pairs, 64 columns
  static constexpr uint32_t COL_O = 192;                    // read + intra output, 16 columns
  static constexpr uint32_t COL_P = 208;                    // P pass, 32 columns
  static constexpr uint32_t TMEM_COLS = 256;                // per team
  static_assert(BYTES <= 232448, "shared memory budget");
};
using DecTc = DecTcT<false>;   // tensor-memory columns (the same for both)

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns into registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 lanes x 32 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// phi(x) and psi(x) = phi(x) - 1 from one exponential (as phi_f32, psi_f32).
__device__ __forceinline__ void phi_psi_f32(float x, float& ph, float& ps) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * 1.4426950408889634f));
  ph = x > 0.f ? x + 1.f : fmaxf(e, 2.16840434e-19f);
  ps = x > 0.f ? x : e - 1.f;
}

// Row t = tid / 8, 16-byte chunk tid % 8 of both 64-feature boxes of the
// group's q, k and v rows (zeros past the last token): r[0..1] q, r[2..3] k,
// r[4..5] v.
__device__ __forceinline__ void load_group_rows(const __nv_bfloat16* qb, const __nv_bfloat16* kb,
                                                const __nv_bfloat16* vb, int t0, int n, int tid, uint4 (&r)[6]) {
  const int t = tid >> 3, ch = tid & 7;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const long long off = (long long)(t0 + t) * DT + 64 * b + 8 * ch;
    const bool valid = t < n;
    r[b] = valid ? *reinterpret_cast<const uint4*>(qb + off) : make_uint4(0u, 0u, 0u, 0u);
    r[2 + b] = valid ? *reinterpret_cast<const uint4*>(kb + off) : make_uint4(0u, 0u, 0u, 0u);
    r[4 + b] = valid ? *reinterpret_cast<const uint4*>(vb + off) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// The bf16 copy of this thread's lane of S^T (fp32 columns COL_S..+127) into
// columns COL_SB..+63, two values per column (lower key index in the low half).
// kScale: the fp32 lane is then multiplied by `scale` in place (decay: the
// held state becomes a^n S before the next group's update adds to it).
template <bool kScale>
__device__ __forceinline__ void refresh_bf16_copy(uint32_t lane_addr, float scale = 1.f) {
#pragma unroll 1
  for (int i0 = 0; i0 < DT; i0 += 32) {
    uint32_t v[32];
    tmem_ld32(lane_addr + DecTc::COL_S + i0, v);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
    tmem_st16(lane_addr + DecTc::COL_SB + i0 / 2, pk);
    if constexpr (kScale) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * scale);
      tmem_st32(lane_addr + DecTc::COL_S + i0, v);
    }
  }
  tmem_st_wait();
}

// Named barrier over the 128 threads of one team (ids 1 and 2; 0 is
// __syncthreads).
__device__ __forceinline__ void team_sync(int team) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + team) : "memory");
}

// Two independent teams of 128 threads per CTA, each taking states
// bh = 2 * cta + team, + 2 * gridDim.x, ...
template <bool kDecay>
__global__ void __launch_bounds__(256, 1)
decode_tc_kernel(float* __restrict__ S, float* __restrict__ z, const __nv_bfloat16* __restrict__ q,
                 const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                 __nv_bfloat16* __restrict__ out, int BH, int ntok, float eps, int* status,
                 const float* __restrict__ alpha, int H) {
  using L = DecTcT<kDecay>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + 2 * L::TEAM_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + 2 * L::TEAM_BYTES + 4);
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(status);
    return;
  }
  const int team = threadIdx.x >> 7;
  const int tid = threadIdx.x & 127;              // thread of the team: lane / value index
  const int warp = tid >> 5;                      // tensor-memory quadrant
  uint8_t* sm = smem_raw + team * L::TEAM_BYTES;
  float* sst = reinterpret_cast<float*>(sm + L::OFF_SST);
  float* zs = reinterpret_cast<float*>(sm + L::OFF_Z);
  float* rden = reinterpret_cast<float*>(sm + L::OFF_DEN);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* bar_p = bar_s + 1;
  uint64_t* bar_mma = bar_s + 2;

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 1);
    mbar_init(bar_mma, 1);
    if (team == 0) *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(tmem_slot, 2 * L::TMEM_COLS);
    tmem_relinquish();
  }
  // constant tiles: ones; P zero (only j < 16 of each row is written later);
  // the psi tiles' rows 16..31 zero except row 18 of psi_hi, ones (rows 16
  // and 17 of psi_hi take z_hi, z_lo in every group)
  {
    uint4* ones = reinterpret_cast<uint4*>(sm + L::OFF_ONES);
    for (int i = tid; i < TTILE / 16; i += 128) ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    uint4* pt = reinterpret_cast<uint4*>(sm + L::OFF_P);
    for (int i = tid; i < TBOX / 16; i += 128) pt[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < 2 * 2 * 16 * 8; i += 128) {
      // (tile, box, row 16..31, chunk)
      const int tile = i >> 8, b = (i >> 7) & 1, r = 16 + ((i >> 3) & 15), ch = i & 7;
      const uint32_t w = (tile == 0 && r == 18) ? 0x3F803F80u : 0u;
      *reinterpret_cast<uint4*>(sm + (tile == 0 ? L::OFF_KH : L::OFF_KL) + b * KBOX + sw128(r, ch)) =
          make_uint4(w, w, w, w);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot + team * L::TMEM_COLS;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);   // lane = tid

  constexpr uint32_t id_read = make_idesc_bf16(128, TG, false, false);   // A (tensor memory), B K-major
  constexpr uint32_t id_p = make_idesc_bf16(128, KROWS, false, false);   // A K-major, B K-major
  constexpr uint32_t id_intra = make_idesc_bf16(128, TG, true, false);   // A MN-major, B K-major
  constexpr uint32_t id_upd = make_idesc_bf16(128, DT, true, true);      // A MN-major, B MN-major
  const uint32_t qa = smem_u32(sm + L::OFF_Q), kha = smem_u32(sm + L::OFF_KH), kla = smem_u32(sm + L::OFF_KL);
  const uint32_t va = smem_u32(sm + L::OFF_V);
  const uint32_t onea = smem_u32(sm + L::OFF_ONES), pa = smem_u32(sm + L::OFF_P);
  const uint32_t qsa = smem_u32(sm + L::OFF_QS), uwa = smem_u32(sm + L::OFF_UW);
  const int ngroups = (ntok + TG - 1) / TG;
  uint32_t ph_s = 0, ph_p = 0, ph_mma = 0;   // phases waited for on each barrier
  uint32_t loads = 0;                        // state loads issued (thread 0 of the team)
  bool ok = true;

  // team 1 starts about half a state later, so that the teams' memory phases
  // alternate instead of coinciding
  if (team == 1) __nanosleep(3000);
  const long long bh0 = 2LL * blockIdx.x + team, bh_step = 2LL * gridDim.x;
  if (tid == 0 && bh0 < BH) {
    // the first state; each later one is loaded while its predecessor runs
    mbar_arrive_expect_tx(bar_s, DT * DT * 4);
    bulk_load(sst, S + bh0 * (long long)(DT * DT), DT * DT * 4, bar_s);
    ++loads;
  }
  // the first group of the next state is prefetched into registers
  uint4 rows[6];
  if (bh0 < BH)
    load_group_rows(q + bh0 * (long long)ntok * DT, k + bh0 * (long long)ntok * DT,
                    v + bh0 * (long long)ntok * DT, 0, min(TG, ntok), tid, rows);
  for (long long bh = bh0; bh < BH && ok; bh += bh_step) {
    float* Sg = S + bh * (long long)(DT * DT);
    const __nv_bfloat16* qb = q + bh * (long long)ntok * DT;
    const __nv_bfloat16* kb = k + bh * (long long)ntok * DT;
    const __nv_bfloat16* vb = v + bh * (long long)ntok * DT;
    __nv_bfloat16* ob = out + bh * (long long)ntok * DT;
    float zr = z[bh * DT + tid];          // z of key index tid
    zs[tid] = zr;
    const float la = kDecay ? log2f(alpha[(int)(bh % H)]) : 0.f;   // log2 a
    team_sync(team);
    for (int g = 0; g < ngroups; ++g) {
      const int t0 = g * TG;
      const int n = min(TG, ntok - t0);
      // ---- the group's tiles: thread tid fills row t = tid / 8, 16-byte
      // chunk ch = tid % 8 of both 64-feature boxes (features 8 ch .. 8 ch + 7
      // and 64 + 8 ch .. 64 + 8 ch + 7); threads of rows 0 and 1 also write
      // z_hi, z_lo (rows 16, 17 of the psi_hi tile)
      if (g > 0) load_group_rows(qb, kb, vb, t0, n, tid, rows);
      {
        const int t = tid >> 3, ch = tid & 7;
        const bool valid = t < n;
        // decay: the read's weight a^(t+1) of query row t and the update's
        // weight w_t = a^(n-1-t) of key row t (0 past the last token)
        const float qsc = kDecay ? exp2f((float)(t + 1) * la) : 1.f;
        const float wt = kDecay && valid ? exp2f((float)(n - 1 - t) * la) : 0.f;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t* pq = reinterpret_cast<const uint32_t*>(&rows[b]);
          const uint32_t* pk = reinterpret_cast<const uint32_t*>(&rows[2 + b]);
          uint4 oq, ok4, ol4, oqs, owh, owl;
          uint32_t* poq = reinterpret_cast<uint32_t*>(&oq);
          uint32_t* pok = reinterpret_cast<uint32_t*>(&ok4);
          uint32_t* pol = reinterpret_cast<uint32_t*>(&ol4);
          uint32_t* pqs = reinterpret_cast<uint32_t*>(&oqs);
          uint32_t* pwh = reinterpret_cast<uint32_t*>(&owh);
          uint32_t* pwl = reinterpret_cast<uint32_t*>(&owl);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float ph0, ps0, ph1, ps1;
            phi_psi_f32(__uint_as_float(pk[h] << 16), ph0, ps0);
            phi_psi_f32(__uint_as_float(pk[h] & 0xFFFF0000u), ph1, ps1);
            const float fq0 = valid ? phi_f32(__uint_as_float(pq[h] << 16)) : 0.f;
            const float fq1 = valid ? phi_f32(__uint_as_float(pq[h] & 0xFFFF0000u)) : 0.f;
            if (!valid) ps0 = ps1 = 0.f;
            poq[h] = pack_bf16x2(fq0, fq1);
            pok[h] = pack_bf16x2(ps0, ps1);
            pol[h] = pack_bf16x2(ps0 - __uint_as_float(pok[h] << 16), ps1 - __uint_as_float(pok[h] & 0xFFFF0000u));
            if constexpr (kDecay) {
              pqs[h] = pack_bf16x2(fq0 * qsc, fq1 * qsc);
              const float x0 = wt * ps0, x1 = wt * ps1;
              pwh[h] = pack_bf16x2(x0, x1);
              pwl[h] = pack_bf16x2(x0 - __uint_as_float(pwh[h] << 16), x1 - __uint_as_float(pwh[h] & 0xFFFF0000u));
            }
          }
          *reinterpret_cast<uint4*>(sm + L::OFF_Q + b * TBOX + sw128(t, ch)) = oq;
          if constexpr (kDecay) {
            // [w_hi], [w_lo] (constant along the row), [w psi]_hi, [w psi]_lo
            const uint32_t whi = pack_bf16x2(wt, wt);
            const float wlo = wt - __uint_as_float(whi << 16);
            const uint32_t wlo2 = pack_bf16x2(wlo, wlo);
            *reinterpret_cast<uint4*>(sm + L::OFF_QS + b * TBOX + sw128(t, ch)) = oqs;
            *reinterpret_cast<uint4*>(sm + L::OFF_ONES + b * TBOX + sw128(t, ch)) = make_uint4(whi, whi, whi, whi);
            *reinterpret_cast<uint4*>(sm + L::OFF_UW + b * TBOX + sw128(t, ch)) = make_uint4(wlo2, wlo2, wlo2, wlo2);
            *reinterpret_cast<uint4*>(sm + L::OFF_UW + TTILE + b * TBOX + sw128(t, ch)) = owh;
            *reinterpret_cast<uint4*>(sm + L::OFF_UW + 2 * TTILE + b * TBOX + sw128(t, ch)) = owl;
          }
          *reinterpret_cast<uint4*>(sm + L::OFF_KH + b * KBOX + sw128(t, ch)) = ok4;
          *reinterpret_cast<uint4*>(sm + L::OFF_KL + b * KBOX + sw128(t, ch)) = ol4;
          *reinterpret_cast<uint4*>(sm + L::OFF_V + b * TBOX + sw128(t, ch)) = rows[4 + b];
          if (t < 2) {
            // z_0 of features 64 b + 8 ch .. + 7: bf16 high part (row 16) or
            // the bf16 remainder (row 17)
            const float4 z0 = *reinterpret_cast<const float4*>(zs + 64 * b + 8 * ch);
            const float4 z1 = *reinterpret_cast<const float4*>(zs + 64 * b + 8 * ch + 4);
            const float zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
            uint4 zw;
            uint32_t* pz = reinterpret_cast<uint32_t*>(&zw);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const uint32_t hi = pack_bf16x2(zz[2 * h], zz[2 * h + 1]);
              pz[h] = t == 0 ? hi
                             : pack_bf16x2(zz[2 * h] - __uint_as_float(hi << 16),
                                           zz[2 * h + 1] - __uint_as_float(hi & 0xFFFF0000u));
            }
            *reinterpret_cast<uint4*>(sm + L::OFF_KH + b * KBOX + sw128(16 + t, ch)) = zw;
          }
        }
      }
      if (g == 0) {
        // the state, loaded while the first group's tiles were built: column
        // tid (S[i][tid], i = 0..127) -> lane tid of S^T, fp32 and the bf16 copy
        ok = mbar_wait(bar_s, ph_s & 1, abort_flag, kTimeoutNs);
        ++ph_s;
        if (!ok) break;
        // (decay: the fp32 state a^n S_0, the copy S_0)
        const float sc0 = kDecay ? exp2f((float)n * la) : 1.f;
#pragma unroll 1
        for (int i0 = 0; i0 < DT; i0 += 32) {
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(sst[(i0 + j) * DT + tid]);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(w[2 * j]), __uint_as_float(w[2 * j + 1]));
          tmem_st16(lane_addr + L::COL_SB + i0 / 2, pk);
          if constexpr (kDecay) {
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(__uint_as_float(w[j]) * sc0);
          }
          tmem_st32(lane_addr + L::COL_S + i0, w);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      team_sync(team);
      // ---- pass 1: the P pass and the read (after the first group's
      // barrier the staging buffer has been read: the next state's load goes
      // into it)
      if (tid == 0) {
        if (g == 0 && bh + bh_step < BH) {
          mbar_arrive_expect_tx(bar_s, DT * DT * 4);
          bulk_load(sst, S + (bh + bh_step) * (long long)(DT * DT), DT * DT * 4, bar_s);
          ++loads;
        }
        tc_fence_after();
        // D_P = phi(Q) [psi_hi ; z_hi ; z_lo ; 1]^T + phi(Q) [psi_lo ; 0]^T;
        // A = phi(Q) K-major read as 128 rows, B K-major 32 rows
#pragma unroll
        for (int kk = 0; kk < DT / 16; ++kk)
          mma_ss(tmem + L::COL_P, make_sdesc(qa + (kk >> 2) * TBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B),
                 make_sdesc(kha + (kk >> 2) * KBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B), id_p, kk > 0);
#pragma unroll
        for (int kk = 0; kk < DT / 16; ++kk)
          mma_ss(tmem + L::COL_P, make_sdesc(qa + (kk >> 2) * TBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B),
                 make_sdesc(kla + (kk >> 2) * KBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B), id_p, 1);
        tc_commit(bar_p);
        // read: D[c][t] = sum_i S^T[c][i] phi(q_t)[i]; A = the bf16 copy in
        // tensor memory (8 columns per K-step of 16), B = phi(Q) K-major
        // (decay: the rows weighted a^(t+1))
        const uint32_t qra = kDecay ? qsa : qa;
#pragma unroll
        for (int kk = 0; kk < DT / 16; ++kk)
          mma_ts(tmem + L::COL_O, tmem + L::COL_SB + kk * 8,
                 make_sdesc(qra + (kk >> 2) * TBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B), id_read, kk > 0);
      }
      ok = mbar_wait(bar_p, ph_p & 1, abort_flag, kTimeoutNs);
      ++ph_p;
      if (!ok) break;
      tc_fence_after();
      // ---- P_tj = D_P[t][j] + s_t masked to j <= t < n (lane t of warp 0),
      // into the K-major B tile; den_t = phi(q_t) . z_0 + sum_j P_tj + eps
      if (warp == 0) {
        uint32_t d[32];
        tmem_ld32(lane_addr + L::COL_P, d);
        tmem_ld_wait();
        const int t = tid;
        if (t < TG) {
          const float st = __uint_as_float(d[18]);
          float pr[16], sum = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            pr[j] = (j <= t && t < n) ? __uint_as_float(d[j]) + st : 0.f;
            if (kDecay) pr[j] *= exp2f((float)(t - j) * la);    // a^(t-j)
            sum += pr[j];
          }
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            uint4 w;
            w.x = pack_bf16x2(pr[8 * c2 + 0], pr[8 * c2 + 1]);
            w.y = pack_bf16x2(pr[8 * c2 + 2], pr[8 * c2 + 3]);
            w.z = pack_bf16x2(pr[8 * c2 + 4], pr[8 * c2 + 5]);
            w.w = pack_bf16x2(pr[8 * c2 + 6], pr[8 * c2 + 7]);
            *reinterpret_cast<uint4*>(sm + L::OFF_P + sw128(t, c2)) = w;
          }
          const float zq = __uint_as_float(d[16]) + __uint_as_float(d[17]);   // phi(q_t) . z_0
          rden[t] = 1.f / ((kDecay ? exp2f((float)(t + 1) * la) * zq : zq) + sum + eps);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      team_sync(team);
      // ---- pass 2: intra-group and the update
      if (tid == 0) {
        tc_fence_after();
        // intra: D[c][t] += sum_j v_j[c] P[t][j]; A = V MN-major (second
        // 64-wide block of c one box on), B = P K-major
        mma_ss(tmem + L::COL_O, make_sdesc(va, TBOX, 1024, kSwizzle128B), make_sdesc(pa, 16, 1024, kSwizzle128B),
               id_intra, 1);
        // update: S^T += V^T 1 + V^T psi_hi + V^T psi_lo (the psi tiles read
        // as MN-major with K = 16: rows 0..15)
        if constexpr (kDecay) {
          // S^T += V^T (w_hi + w_lo + [w psi]_hi + [w psi]_lo), on a^n S_0
#pragma unroll
          for (int u = 0; u < 4; ++u)
            mma_ss(tmem + L::COL_S, make_sdesc(va, TBOX, 1024, kSwizzle128B),
                   make_sdesc(u == 0 ? onea : uwa + (u - 1) * TTILE, TBOX, 1024, kSwizzle128B), id_upd, 1);
        } else {
          mma_ss(tmem + L::COL_S, make_sdesc(va, TBOX, 1024, kSwizzle128B), make_sdesc(kha, KBOX, 1024, kSwizzle128B),
                 id_upd, 1);
          mma_ss(tmem + L::COL_S, make_sdesc(va, TBOX, 1024, kSwizzle128B), make_sdesc(kla, KBOX, 1024, kSwizzle128B),
                 id_upd, 1);
          mma_ss(tmem + L::COL_S, make_sdesc(va, TBOX, 1024, kSwizzle128B),
                 make_sdesc(onea, TBOX, 1024, kSwizzle128B), id_upd, 1);
        }
        tc_commit(bar_mma);
      }
      ok = mbar_wait(bar_mma, ph_mma & 1, abort_flag, kTimeoutNs);
      ++ph_mma;
      if (!ok) break;
      tc_fence_after();
      // ---- outputs out[t0 + t][tid] = D[tid][t] / den_t
      {
        uint32_t o[16];
        tmem_ld16(lane_addr + L::COL_O, o);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < TG; ++t)
          if (t < n) ob[(long long)(t0 + t) * DT + tid] = __float2bfloat16_rn(__uint_as_float(o[t]) * rden[t]);
      }
      // z of key index tid: the n tokens' 1 and their psi (hi + lo)
      {
        const uint8_t* hb = sm + L::OFF_KH + (tid >> 6) * KBOX;
        const uint8_t* lb = sm + L::OFF_KL + (tid >> 6) * KBOX;
        const int ch = (tid & 63) >> 3, pos = tid & 7;
        float acc = kDecay ? 0.f : (float)n;
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          const uint32_t off = sw128(t, ch) + 2 * pos;
          const float ps = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(hb + off)) +
                           __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(lb + off));
          if (kDecay)
            acc += t < n ? exp2f((float)(n - 1 - t) * la) * (1.f + ps) : 0.f;   // w_t phi(k_t)
          else
            acc += ps;
        }
        zr = kDecay ? exp2f((float)n * la) * zr + acc : zr + acc;
      }
      // the next group reads the updated state through its bf16 copy
      if (g + 1 < ngroups) {
        if constexpr (kDecay)
          refresh_bf16_copy<true>(lane_addr, exp2f((float)min(TG, ntok - t0 - TG) * la));   // a^(next n)
        else
          refresh_bf16_copy<false>(lane_addr);
      }
      tc_fence_before();
      team_sync(team);    // tiles, rden and zs are rewritten next
      zs[tid] = zr;
      team_sync(team);
    }
    if (!ok) break;
    // the next state's first group, in flight during the store
    if (bh + bh_step < BH)
      load_group_rows(q + (bh + bh_step) * (long long)ntok * DT, k + (bh + bh_step) * (long long)ntok * DT,
                      v + (bh + bh_step) * (long long)ntok * DT, 0, min(TG, ntok), tid, rows);
    // S^T lane tid -> column tid of the state in global memory: for each key
    // index i a warp writes 32 consecutive values of row i
#pragma unroll 1
    for (int i0 = 0; i0 < DT; i0 += 32) {
      uint32_t w[32];
      tmem_ld32(lane_addr + L::COL_S + i0, w);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) Sg[(i0 + j) * DT + tid] = __uint_as_float(w[j]);
    }
    z[bh * DT + tid] = zr;
    // tensor memory is rewritten by the next state's transposition
    tc_fence_before();
    team_sync(team);
  }
  // ---------------- teardown ----------------
  if (tid == 0) {
    // nothing in flight once shared and tensor memory are released: a state
    // load issued but not waited for (abort path), the last MMA passes
    if (loads > ph_s) mbar_drain(bar_s, ph_s & 1, kTimeoutNs);
    if (ph_p > 0) mbar_drain(bar_p, (ph_p - 1) & 1, kTimeoutNs);
    if (ph_mma > 0) mbar_drain(bar_mma, (ph_mma - 1) & 1, kTimeoutNs);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) report_timeout(status);
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, 2 * L::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Delta rule ("Linear Attention, 곱의 순서를 바꾸면 생기는 일", paragraph on 델타
// 규칙): u_t = S_{t-1}^T k_t, S_t = S_{t-1} + k_t (v_t - u_t)^T, out_t = S_t^T q_t,
// keys and queries as given. Over a group of n tokens from S_0 the increments
// u'_t = v_t - S_{t-1}^T k_t solve the unit lower-triangular system
//   u'_t = v_t - S_0^T k_t - sum_{j < t} (k_t . k_j) u'_j,
// and out_t = S_0^T q_t + sum_{j <= t} (q_t . k_j) u'_j, S_n = S_0 + sum_t k_t u'_t^T.
// Per group:
//   MMA      D_P[r][j] = [K ; Q]_r . k_j        (pair products, exact in fp32)
//   MMA x 2  D[c][r] = S^T [K ; Q]^T            (the state as bf16 hi, then lo:
//                                               about 16 bits, since the
//                                               correction v - S^T k needs them)
//   lane c   the 16-step forward substitution for u'[c][.] and the outputs
//   MMA x 2  S^T += U'^T K                      (U' as bf16 hi + lo in tensor memory)
// Two teams per CTA as the kernel above; no z.
// ---------------------------------------------------------------------------
constexpr int DROWS = 32;                // rows of the [K ; Q] tile
constexpr int DBOX = DROWS * 128;        // bytes of one [32 rows][64 bf16] SW128 box

struct DecDelta {
  static constexpr int OFF_SST = 0;                         // fp32 [128][128] state (bulk load)
  static constexpr int OFF_KQ = OFF_SST + DT * DT * 4;      // [K ; Q] bf16, K-major, two boxes
  static constexpr int OFF_A = OFF_KQ + 2 * DBOX;           // fp32 [16][16] k_t . k_j
  static constexpr int OFF_QK = OFF_A + TG * TG * 4;        // fp32 [16][16] q_t . k_j
  static constexpr int OFF_BAR = OFF_QK + TG * TG * 4;      // 4 mbarriers
  // the pair-product MMA reads [K ; Q] as 128 rows (rows 32.. are whatever
  // follows; their results are not read): inside the team's region
  static constexpr int TEAM_BYTES =
      ((OFF_BAR + 32 > OFF_KQ + DBOX + 16 * 1024 ? OFF_BAR + 32 : OFF_KQ + DBOX + 16 * 1024) + 1023) / 1024 * 1024;
  static constexpr int BYTES = 2 * TEAM_BYTES + 16;
  static_assert(OFF_KQ % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
  static_assert(BYTES <= 232448, "shared memory budget");
  // tensor memory columns (per team)
  static constexpr uint32_t COL_S = 0;                      // S^T fp32, 128 columns
  static constexpr uint32_t COL_SB = 128;                   // S^T bf16 (hi, then lo), 64 columns
  static constexpr uint32_t COL_KQ = 192;                   // S^T [K ; Q]^T, 32 columns
  static constexpr uint32_t COL_P = 224;                    // pair products, 16 columns
  static constexpr uint32_t COL_U = 240;                    // U' bf16 hi (8) and lo (8)
  static constexpr uint32_t TMEM_COLS = 256;
};

// The remainder S - bf16(S) of this thread's lane of S^T, as bf16, into the
// copy columns (the high part's read has finished).
__device__ __forceinline__ void lo_copy(uint32_t lane_addr) {
#pragma unroll 1
  for (int i0 = 0; i0 < DT; i0 += 32) {
    uint32_t v[32];
    tmem_ld32(lane_addr + DecDelta::COL_S + i0, v);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float a = __uint_as_float(v[2 * j]), b = __uint_as_float(v[2 * j + 1]);
      const uint32_t hi = pack_bf16x2(a, b);
      pk[j] = pack_bf16x2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
    }
    tmem_st16(lane_addr + DecDelta::COL_SB + i0 / 2, pk);
  }
  tmem_st_wait();
}

__global__ void __launch_bounds__(256, 1)
decode_tc_delta_kernel(float* __restrict__ S, const __nv_bfloat16* __restrict__ q,
                       const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                       __nv_bfloat16* __restrict__ out, int BH, int ntok, int* status) {
  using L = DecDelta;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + 2 * L::TEAM_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + 2 * L::TEAM_BYTES + 4);
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(status);
    return;
  }
  const int team = threadIdx.x >> 7;
  const int tid = threadIdx.x & 127;              // thread of the team: lane / value index
  const int warp = tid >> 5;
  uint8_t* sm = smem_raw + team * L::TEAM_BYTES;
  float* sst = reinterpret_cast<float*>(sm + L::OFF_SST);
  float* sA = reinterpret_cast<float*>(sm + L::OFF_A);
  float* sQK = reinterpret_cast<float*>(sm + L::OFF_QK);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* bar_r = bar_s + 1;
  uint64_t* bar_mma = bar_s + 2;

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_r, 1);
    mbar_init(bar_mma, 1);
    if (team == 0) *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(tmem_slot, 2 * L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot + team * L::TMEM_COLS;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);   // lane = tid

  constexpr uint32_t id_pair = make_idesc_bf16(128, TG, false, false);     // A, B K-major (smem)
  constexpr uint32_t id_read = make_idesc_bf16(128, DROWS, false, false);  // A tensor memory, B K-major
  constexpr uint32_t id_upd = make_idesc_bf16(128, DT, false, true);       // A tensor memory, B MN-major
  const uint32_t kqa = smem_u32(sm + L::OFF_KQ);
  const int ngroups = (ntok + TG - 1) / TG;
  uint32_t ph_s = 0, ph_r = 0, ph_mma = 0;
  uint32_t loads = 0;
  bool ok = true;

  if (team == 1) __nanosleep(3000);
  const long long bh0 = 2LL * blockIdx.x + team, bh_step = 2LL * gridDim.x;
  if (tid == 0 && bh0 < BH) {
    mbar_arrive_expect_tx(bar_s, DT * DT * 4);
    bulk_load(sst, S + bh0 * (long long)(DT * DT), DT * DT * 4, bar_s);
    ++loads;
  }
  for (long long bh = bh0; bh < BH && ok; bh += bh_step) {
    float* Sg = S + bh * (long long)(DT * DT);
    const __nv_bfloat16* qb = q + bh * (long long)ntok * DT;
    const __nv_bfloat16* kb = k + bh * (long long)ntok * DT;
    const __nv_bfloat16* vb = v + bh * (long long)ntok * DT;
    __nv_bfloat16* ob = out + bh * (long long)ntok * DT;
    for (int g = 0; g < ngroups; ++g) {
      const int t0 = g * TG;
      const int n = min(TG, ntok - t0);
      // ---- [K ; Q] tile: thread tid fills row t = tid / 8 (k_t) and row
      // 16 + t (q_t), 16-byte chunk tid % 8 of both boxes; zeros past n.
      // Lane tid's values v_t[tid] for the substitution.
      {
        const int t = tid >> 3, ch = tid & 7;
        const bool valid = t < n;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const long long off = (long long)(t0 + t) * DT + 64 * b + 8 * ch;
          const uint4 kk = valid ? *reinterpret_cast<const uint4*>(kb + off) : make_uint4(0u, 0u, 0u, 0u);
          const uint4 qq = valid ? *reinterpret_cast<const uint4*>(qb + off) : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(sm + L::OFF_KQ + b * DBOX + sw128(t, ch)) = kk;
          *reinterpret_cast<uint4*>(sm + L::OFF_KQ + b * DBOX + sw128(16 + t, ch)) = qq;
        }
      }
      float vr[TG];
#pragma unroll
      for (int t = 0; t < TG; ++t)
        vr[t] = t < n ? __bfloat162float(vb[(long long)(t0 + t) * DT + tid]) : 0.f;
      if (g == 0) {
        // the state: column tid of S -> lane tid of S^T, fp32 and the bf16 high part
        ok = mbar_wait(bar_s, ph_s & 1, abort_flag, kTimeoutNs);
        ++ph_s;
        if (!ok) break;
#pragma unroll 1
        for (int i0 = 0; i0 < DT; i0 += 32) {
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(sst[(i0 + j) * DT + tid]);
          tmem_st32(lane_addr + L::COL_S + i0, w);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(w[2 * j]), __uint_as_float(w[2 * j + 1]));
          tmem_st16(lane_addr + L::COL_SB + i0 / 2, pk);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      team_sync(team);
      // ---- pair products and the read with the high part
      if (tid == 0) {
        if (g == 0 && bh + bh_step < BH) {
          mbar_arrive_expect_tx(bar_s, DT * DT * 4);
          bulk_load(sst, S + (bh + bh_step) * (long long)(DT * DT), DT * DT * 4, bar_s);
          ++loads;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DT / 16; ++kk) {
          const uint64_t d = make_sdesc(kqa + (kk >> 2) * DBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          mma_ss(tmem + L::COL_P, d, d, id_pair, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DT / 16; ++kk)
          mma_ts(tmem + L::COL_KQ, tmem + L::COL_SB + kk * 8,
                 make_sdesc(kqa + (kk >> 2) * DBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B), id_read, kk > 0);
        tc_commit(bar_r);
      }
      ok = mbar_wait(bar_r, ph_r & 1, abort_flag, kTimeoutNs);
      ++ph_r;
      if (!ok) break;
      tc_fence_after();
      // ---- the low part of the state into the copy; warp 0 moves the pair
      // products to shared memory (row r < 16: k_r . k_j; row 16 + t: q_t . k_j)
      lo_copy(lane_addr);
      if (warp == 0) {
        uint32_t d[16];
        tmem_ld16(lane_addr + L::COL_P, d);
        tmem_ld_wait();
        float* dst = tid < TG ? sA + tid * TG : sQK + (tid - TG) * TG;
#pragma unroll
        for (int j = 0; j < TG; ++j) dst[j] = __uint_as_float(d[j]);
      }
      tc_fence_before();
      team_sync(team);
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DT / 16; ++kk)
          mma_ts(tmem + L::COL_KQ, tmem + L::COL_SB + kk * 8,
                 make_sdesc(kqa + (kk >> 2) * DBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B), id_read, 1);
        tc_commit(bar_r);
      }
      ok = mbar_wait(bar_r, ph_r & 1, abort_flag, kTimeoutNs);
      ++ph_r;
      if (!ok) break;
      tc_fence_after();
      // ---- lane tid: u'_t = v_t - (S^T k_t) - sum_{j<t} (k_t . k_j) u'_j,
      // out_t = (S^T q_t) + sum_{j<=t} (q_t . k_j) u'_j
      {
        uint32_t d[32];
        tmem_ld32(lane_addr + L::COL_KQ, d);
        tmem_ld_wait();
        float u[TG];
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          float x = vr[t] - __uint_as_float(d[t]);
#pragma unroll
          for (int j = 0; j < t; ++j) x = fmaf(-sA[t * TG + j], u[j], x);
          u[t] = t < n ? x : 0.f;
        }
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          float o = __uint_as_float(d[TG + t]);
#pragma unroll
          for (int j = 0; j <= t; ++j) o = fmaf(sQK[t * TG + j], u[j], o);
          if (t < n) ob[(long long)(t0 + t) * DT + tid] = __float2bfloat16_rn(o);
        }
        // U' as bf16 hi (columns COL_U..+7) and lo (COL_U+8..+15), token
        // pairs per column (lower token in the low half)
        uint32_t pu[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          pu[j] = pack_bf16x2(u[2 * j], u[2 * j + 1]);
          pu[8 + j] = pack_bf16x2(u[2 * j] - __uint_as_float(pu[j] << 16),
                                  u[2 * j + 1] - __uint_as_float(pu[j] & 0xFFFF0000u));
        }
        tmem_st16(lane_addr + L::COL_U, pu);
        tmem_st_wait();
      }
      tc_fence_before();
      team_sync(team);
      // ---- update: S^T += U'_hi K + U'_lo K (K = 16 tokens, B = the K rows
      // of the tile read MN-major)
      if (tid == 0) {
        tc_fence_after();
        mma_ts(tmem + L::COL_S, tmem + L::COL_U, make_sdesc(kqa, DBOX, 1024, kSwizzle128B), id_upd, 1);
        mma_ts(tmem + L::COL_S, tmem + L::COL_U + 8, make_sdesc(kqa, DBOX, 1024, kSwizzle128B), id_upd, 1);
        tc_commit(bar_mma);
      }
      ok = mbar_wait(bar_mma, ph_mma & 1, abort_flag, kTimeoutNs);
      ++ph_mma;
      if (!ok) break;
      tc_fence_after();
      if (g + 1 < ngroups) refresh_bf16_copy<false>(lane_addr);
      tc_fence_before();
      team_sync(team);    // the tile and the pair products are rewritten next
    }
    if (!ok) break;
#pragma unroll 1
    for (int i0 = 0; i0 < DT; i0 += 32) {
      uint32_t w[32];
      tmem_ld32(lane_addr + L::COL_S + i0, w);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) Sg[(i0 + j) * DT + tid] = __uint_as_float(w[j]);
    }
    tc_fence_before();
    team_sync(team);
  }
  // ---------------- teardown ----------------
  if (tid == 0) {
    if (loads > ph_s) mbar_drain(bar_s, ph_s & 1, kTimeoutNs);
    if (ph_r > 0) mbar_drain(bar_r, (ph_r - 1) & 1, kTimeoutNs);
    if (ph_mma > 0) mbar_drain(bar_mma, (ph_mma - 1) & 1, kTimeoutNs);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) report_timeout(status);
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, 2 * L::TMEM_COLS);
  }
}

}  // namespace

bool tc_decode_supported(int dk, int dv, la_dtype dtype, int ntok) {
  return dtype == LA_BF16 && dk == DT && dv == DT && ntok >= 2;
}

template <bool kDecay>
cudaError_t launch_decode_tc(const DecodeArgs& a, const float* alpha = nullptr, int H = 1) {
  constexpr int smem = DecTcT<kDecay>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<kDecay>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // two states at a time per CTA (one per team), one CTA per SM
  const int ctas = (int)std::min<long long>((a.BH + 1) / 2, (long long)sms);
  decode_tc_kernel<kDecay><<<ctas, 256, smem, a.stream>>>(
      a.S, a.z, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
      (__nv_bfloat16*)a.out, a.BH, a.ntok, a.eps, device_status_ptr(), alpha, H);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t tc_decode_steps(const DecodeArgs& a) { return launch_decode_tc<false>(a); }

cudaError_t tc_decode_steps_decay(const DecodeArgs& a, const float* alpha, int H) {
  return launch_decode_tc<true>(a, alpha, H);
}

cudaError_t tc_decode_steps_delta(const DecodeArgs& a) {
  constexpr int smem = DecDelta::BYTES;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_delta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int ctas = (int)std::min<long long>((a.BH + 1) / 2, (long long)sms);
  decode_tc_delta_kernel<<<ctas, 256, smem, a.stream>>>(
      a.S, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v, (__nv_bfloat16*)a.out,
      a.BH, a.ntok, device_status_ptr());
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace la
