// Multi-token decode on the tensor cores (bf16 tokens, dk = dv = 128, fp32
// state): T consecutive tokens of one (batch, head) per CTA, in groups of up
// to TG = 16, the state read and written once per call.
//
// The recurrence ("Linear Attention: KV를 고정 크기 상태에 누적하기", section
// "상태 갱신과 읽기를 식으로 정리하기") over a group of n tokens starting from
// S_0, z_0, in its chunked form (the masked sums of "상태공간모델·선형
// 어텐션", section 2, re-associated):
//   num_t = S_0^T phi(q_t) + sum_{j <= t} (phi(q_t) . phi(k_j)) v_j
//   den_t = phi(q_t) . z_0 + sum_{j <= t} phi(q_t) . phi(k_j) + eps
//   S    <- S_0 + sum_j phi(k_j) v_j^T,   z <- z_0 + sum_j phi(k_j)
// The state is held transposed in tensor memory, S^T (lane = value index c,
// column = key index i), in fp32, with a bf16 copy of it beside (two values
// per column). Per group, four MMAs (M = 128):
//   read    D[c][t]  = S^T (bf16 copy, tensor memory) x phi(Q)^T   N = 16, K = 128
//   intra   D[c][t] += V^T P^T, P = (phi(Q) phi(K)^T) masked j <= t  N = 16, K = 16
//   update  S^T     += V^T 1 + V^T psi_hi(K) + V^T psi_lo(K)         N = 128, K = 16
// with psi = phi - 1 = psi_hi + psi_lo (two bf16 parts): the update carries
// the large common part of phi(k) (its 1) exactly (V^T times a tile of ones)
// and psi to about 16 bits, so the state keeps fp32 accuracy; the read rounds
// the state and phi(q) to bf16, as the chunked forward does.
// P (fp32 dot products of the fp32 features), the denominators and z are on
// the CUDA cores in fp32.
//
// One CTA of 128 threads per (b, h), two CTAs per SM (256 tensor-memory
// columns, ~104 KB of shared memory each). Thread c (warp c / 32) owns lane
// c: value index c of the state and of the outputs, key index c of z. The
// state moves between global and shared memory as one 64 KB bulk copy each
// way; thread c reads or writes column c of the shared copy (consecutive
// addresses across a warp). Every wait is bounded; on a timeout the CTA stops
// and reports through the device status word.
#include "la_tc_common.cuh"

namespace la {

namespace {

using namespace sm100;

constexpr int DT = 128;                 // dk = dv
constexpr int TG = 16;                  // tokens per group
constexpr int TBOX = TG * 128;          // bytes of one [16 rows][64 bf16] SW128 box
constexpr int TTILE = 2 * TBOX;         // a [16][128] bf16 tile (two boxes)

struct DecTc {
  static constexpr int OFF_SST = 0;                         // fp32 [128][128] state copy (bulk in / out)
  static constexpr int OFF_Q = OFF_SST + DT * DT * 4;       // phi(Q) bf16, K-major [t][i]
  static constexpr int OFF_K = OFF_Q + TTILE;               // psi(K) bf16 high part, MN-major [t][i]
  static constexpr int OFF_KL = OFF_K + TTILE;              // psi(K) bf16 low part, MN-major [t][i]
  static constexpr int OFF_V = OFF_KL + TTILE;              // V bf16, MN-major [t][c]
  static constexpr int OFF_ONES = OFF_V + TTILE;            // ones, MN-major [t][i]
  static constexpr int OFF_P = OFF_ONES + TTILE;            // P bf16, K-major [t][j] (j < 16 used)
  static constexpr int FROW = DT + 1;                       // padded fp32 feature rows (no bank conflicts)
  static constexpr int OFF_FQ = OFF_P + TBOX;               // fp32 phi(q) [16][FROW]
  static constexpr int OFF_FK = OFF_FQ + TG * FROW * 4;     // fp32 phi(k) [16][FROW] (0 past the group)
  static constexpr int OFF_PF = OFF_FK + TG * FROW * 4;     // fp32 P [16][16]
  static constexpr int OFF_Z = OFF_PF + TG * TG * 4;        // fp32 z [128]
  static constexpr int OFF_DEN = OFF_Z + DT * 4;            // fp32 1 / den [16]
  static constexpr int OFF_BAR = OFF_DEN + TG * 4;          // 2 mbarriers
  static constexpr int OFF_MISC = OFF_BAR + 16;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(OFF_Q % 1024 == 0 && OFF_KL % 1024 == 0 && OFF_P % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
  // tensor memory columns
  static constexpr uint32_t COL_S = 0;                      // S^T fp32, 128 columns
  static constexpr uint32_t COL_SB = 128;                   // S^T bf16 pairs, 64 columns
  static constexpr uint32_t COL_O = 192;                    // read/intra output, 16 columns
  static constexpr uint32_t TMEM_COLS = 256;
};

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(smem_src)),
               "r"(bytes)
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

// The bf16 copy of this thread's lane of S^T (fp32 columns COL_S..+127) into
// columns COL_SB..+63, two values per column (lower key index in the low half).
__device__ __forceinline__ void refresh_bf16_copy(uint32_t lane_addr) {
#pragma unroll 1
  for (int i0 = 0; i0 < DT; i0 += 32) {
    uint32_t v[32];
    tmem_ld32(lane_addr + DecTc::COL_S + i0, v);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
    tmem_st16(lane_addr + DecTc::COL_SB + i0 / 2, pk);
  }
  tmem_st_wait();
}

__global__ void __launch_bounds__(128, 2)
decode_tc_kernel(float* __restrict__ S, float* __restrict__ z, const __nv_bfloat16* __restrict__ q,
                 const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                 __nv_bfloat16* __restrict__ out, int ntok, float eps, int* status) {
  using L = DecTc;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  float* sst = reinterpret_cast<float*>(sm + L::OFF_SST);
  float* fq = reinterpret_cast<float*>(sm + L::OFF_FQ);
  float* fk = reinterpret_cast<float*>(sm + L::OFF_FK);
  float* pf = reinterpret_cast<float*>(sm + L::OFF_PF);
  float* zs = reinterpret_cast<float*>(sm + L::OFF_Z);
  float* rden = reinterpret_cast<float*>(sm + L::OFF_DEN);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* bar_mma = bar_s + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::OFF_MISC + 4);
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) report_timeout(status);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5;
  const long long bh = blockIdx.x;
  float* Sg = S + bh * (long long)(DT * DT);
  const __nv_bfloat16* qb = q + bh * (long long)ntok * DT;
  const __nv_bfloat16* kb = k + bh * (long long)ntok * DT;
  const __nv_bfloat16* vb = v + bh * (long long)ntok * DT;
  __nv_bfloat16* ob = out + bh * (long long)ntok * DT;

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  // the ones tile (every element 1.0)
  {
    uint4* ones = reinterpret_cast<uint4*>(sm + L::OFF_ONES);
    for (int i = tid; i < TTILE / 16; i += 128) ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);   // lane = tid

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_s, DT * DT * 4);
    bulk_load(sst, Sg, DT * DT * 4, bar_s);
  }
  float zr = z[bh * DT + tid];            // z of key index tid
  zs[tid] = zr;
  bool ok = mbar_wait(bar_s, 0, abort_flag, kTimeoutNs);
  if (ok) {
    // column tid of the state (S[i][tid], i = 0..127) -> lane tid of S^T,
    // fp32 and the bf16 copy
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
  constexpr uint32_t id_read = make_idesc_bf16(128, TG, false, false);   // A (tensor memory), B K-major
  constexpr uint32_t id_intra = make_idesc_bf16(128, TG, true, false);   // A MN-major, B K-major
  constexpr uint32_t id_upd = make_idesc_bf16(128, DT, true, true);      // A MN-major, B MN-major
  const uint32_t qa = smem_u32(sm + L::OFF_Q), ka = smem_u32(sm + L::OFF_K), kla = smem_u32(sm + L::OFF_KL);
  const uint32_t va = smem_u32(sm + L::OFF_V);
  const uint32_t onea = smem_u32(sm + L::OFF_ONES), pa = smem_u32(sm + L::OFF_P);

  const int ngroups = (ntok + TG - 1) / TG;
  int issued = 0;                         // groups whose MMAs thread 0 issued
  for (int g = 0; g < ngroups && ok; ++g) {
    const int t0 = g * TG;
    const int n = min(TG, ntok - t0);
    // ---- the group's tiles: thread tid fills row t = tid / 8, 16-byte chunk
    // ch = tid % 8 of both 64-feature boxes (features 8 ch .. 8 ch + 7 and
    // 64 + 8 ch .. 64 + 8 ch + 7)
    {
      const int t = tid >> 3, ch = tid & 7;
      const bool valid = t < n;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int f0 = 64 * b + 8 * ch;
        uint4 wq = make_uint4(0u, 0u, 0u, 0u), wk = wq, wv = wq;
        if (valid) {
          wq = *reinterpret_cast<const uint4*>(qb + (long long)(t0 + t) * DT + f0);
          wk = *reinterpret_cast<const uint4*>(kb + (long long)(t0 + t) * DT + f0);
          wv = *reinterpret_cast<const uint4*>(vb + (long long)(t0 + t) * DT + f0);
        }
        const uint32_t* pq = reinterpret_cast<const uint32_t*>(&wq);
        const uint32_t* pk = reinterpret_cast<const uint32_t*>(&wk);
        uint4 oq, ok4, ol4;
        uint32_t* poq = reinterpret_cast<uint32_t*>(&oq);
        uint32_t* pok = reinterpret_cast<uint32_t*>(&ok4);
        uint32_t* pol = reinterpret_cast<uint32_t*>(&ol4);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float q0 = __uint_as_float(pq[h] << 16), q1 = __uint_as_float(pq[h] & 0xFFFF0000u);
          const float k0 = __uint_as_float(pk[h] << 16), k1 = __uint_as_float(pk[h] & 0xFFFF0000u);
          const float fq0 = valid ? phi_f32(q0) : 0.f, fq1 = valid ? phi_f32(q1) : 0.f;
          const float fk0 = valid ? phi_f32(k0) : 0.f, fk1 = valid ? phi_f32(k1) : 0.f;
          const float sk0 = valid ? psi_f32(k0) : 0.f, sk1 = valid ? psi_f32(k1) : 0.f;
          fq[t * L::FROW + f0 + 2 * h] = fq0;
          fq[t * L::FROW + f0 + 2 * h + 1] = fq1;
          fk[t * L::FROW + f0 + 2 * h] = fk0;
          fk[t * L::FROW + f0 + 2 * h + 1] = fk1;
          poq[h] = pack_bf16x2(fq0, fq1);
          pok[h] = pack_bf16x2(sk0, sk1);
          pol[h] = pack_bf16x2(sk0 - __uint_as_float(pok[h] << 16), sk1 - __uint_as_float(pok[h] & 0xFFFF0000u));
        }
        const uint32_t off = b * TBOX + sw128(t, ch);
        *reinterpret_cast<uint4*>(sm + L::OFF_Q + off) = oq;
        *reinterpret_cast<uint4*>(sm + L::OFF_K + off) = ok4;
        *reinterpret_cast<uint4*>(sm + L::OFF_KL + off) = ol4;
        *reinterpret_cast<uint4*>(sm + L::OFF_V + off) = wv;
      }
    }
    __syncthreads();
    // ---- P[t][j] = phi(q_t) . phi(k_j) (fp32), masked to j <= t < n; thread
    // tid computes (t, j) = (tid / 16, tid % 16) and (tid / 16 + 8, tid % 16)
    {
      const int j = tid & 15;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = (tid >> 4) + 8 * h;
        float dot = 0.f;
        if (j <= t && t < n) {
#pragma unroll 8
          for (int i = 0; i < DT; ++i) dot = fmaf(fq[t * L::FROW + i], fk[j * L::FROW + i], dot);
        }
        pf[t * TG + j] = dot;
      }
    }
    __syncthreads();
    // ---- P in bf16 as the K-major B tile ([t][j], j < 16 of a 64-wide box;
    // the rest of the box stays zero: it is never read, K = 16); the
    // denominators 1 / (phi(q_t) . z_0 + sum_j P[t][j] + eps)
    {
      const int t = tid >> 3, ch = tid & 7;   // 16 rows x 8 chunks: chunks 0, 1 hold j < 16
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (ch < 2) {
        const float* pr = pf + t * TG + 8 * ch;
        w.x = pack_bf16x2(pr[0], pr[1]);
        w.y = pack_bf16x2(pr[2], pr[3]);
        w.z = pack_bf16x2(pr[4], pr[5]);
        w.w = pack_bf16x2(pr[6], pr[7]);
      }
      *reinterpret_cast<uint4*>(sm + L::OFF_P + sw128(t, ch)) = w;
      if (tid < TG) {
        float d = eps;
#pragma unroll 4
        for (int i = 0; i < DT; ++i) d = fmaf(fq[tid * L::FROW + i], zs[i], d);
#pragma unroll
        for (int jj = 0; jj < TG; ++jj) d += pf[tid * TG + jj];
        rden[tid] = 1.f / d;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- the group's MMAs
    if (tid == 0) {
      tc_fence_after();
      // read: D[c][t] = sum_i S^T[c][i] phi(q_t)[i]; A = the bf16 copy in
      // tensor memory (8 columns per K-step of 16), B = phi(Q) K-major
#pragma unroll
      for (int kk = 0; kk < DT / 16; ++kk)
        mma_ts(tmem + L::COL_O, tmem + L::COL_SB + kk * 8,
               make_sdesc(qa + (kk >> 2) * TBOX + (kk & 3) * 32, 16, 1024, kSwizzle128B), id_read, kk > 0);
      // intra: D[c][t] += sum_j v_j[c] P[t][j]; A = V MN-major (second
      // 64-wide block of c one box on), B = P K-major
      mma_ss(tmem + L::COL_O, make_sdesc(va, TBOX, 1024, kSwizzle128B), make_sdesc(pa, 16, 1024, kSwizzle128B),
             id_intra, 1);
      // update: S^T += V^T 1 + V^T psi_hi(K) + V^T psi_lo(K) (after the read
      // in issue order)
      mma_ss(tmem + L::COL_S, make_sdesc(va, TBOX, 1024, kSwizzle128B), make_sdesc(ka, TBOX, 1024, kSwizzle128B),
             id_upd, 1);
      mma_ss(tmem + L::COL_S, make_sdesc(va, TBOX, 1024, kSwizzle128B), make_sdesc(kla, TBOX, 1024, kSwizzle128B),
             id_upd, 1);
      mma_ss(tmem + L::COL_S, make_sdesc(va, TBOX, 1024, kSwizzle128B), make_sdesc(onea, TBOX, 1024, kSwizzle128B),
             id_upd, 1);
      tc_commit(bar_mma);
      issued = g + 1;
    }
    ok = mbar_wait(bar_mma, g & 1, abort_flag, kTimeoutNs);
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
    // z of key index tid, fp32 exact
#pragma unroll 4
    for (int t = 0; t < TG; ++t) zr += fk[t * L::FROW + tid];
    // the next group reads the updated state through its bf16 copy
    if (g + 1 < ngroups) refresh_bf16_copy(lane_addr);
    tc_fence_before();
    __syncthreads();    // tiles, fq/fk/pf, rden and zs are rewritten next
    zs[tid] = zr;
  }
  if (ok) {
    // S^T lane tid -> column tid of the shared copy -> one bulk store
#pragma unroll 1
    for (int i0 = 0; i0 < DT; i0 += 32) {
      uint32_t w[32];
      tmem_ld32(lane_addr + L::COL_S + i0, w);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) sst[(i0 + j) * DT + tid] = __uint_as_float(w[j]);
    }
    z[bh * DT + tid] = zr;
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (ok && tid == 0) {
    bulk_store(Sg, sst, DT * DT * 4);
    tma_store_commit();
    tma_store_wait<0>();
  }
  // ---------------- teardown ----------------
  if (tid == 0) {
    // nothing in flight once shared and tensor memory are released: the
    // state load and the last group's MMAs (also on the abort path)
    mbar_drain(bar_s, 0, kTimeoutNs);
    if (issued > 0) mbar_drain(bar_mma, (issued - 1) & 1, kTimeoutNs);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) report_timeout(status);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

}  // namespace

bool tc_decode_supported(int dk, int dv, la_dtype dtype, int ntok) {
  return dtype == LA_BF16 && dk == DT && dv == DT && ntok >= 2;
}

cudaError_t tc_decode_steps(const DecodeArgs& a) {
  constexpr int smem = DecTc::BYTES;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<<<a.BH, 128, smem, a.stream>>>(a.S, a.z, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k,
                                                  (const __nv_bfloat16*)a.v, (__nv_bfloat16*)a.out, a.ntok, a.eps,
                                                  device_status_ptr());
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace la
