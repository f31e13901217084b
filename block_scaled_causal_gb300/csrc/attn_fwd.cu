// Leak-free causal MXFP8 attention forward for sm_103a (tcgen05 / TMEM / TMA).
//
// "[PyTorch] Add causal MXFP8 attention without future-token leakage through V scales"
// (TransformerEngine PR #3865), Description:
//   * keys in completed 32-token blocks (j < 32*floor(i/32)) are attended in MXFP8 with V quantised
//     columnwise (one scale per 32 consecutive tokens), so every V scale read covers visible tokens;
//   * the query's own block (at most 32 keys, j <= i) is attended on the token-normalised V copy;
//   * the two partials are merged through their log-sum-exps.
// Here both key sets share one running softmax (max m and sum l) per row, which is the same merge
// done incrementally, and both P.V products accumulate into one fp32 O accumulator in TMEM.
//
// One CTA computes one 128-row query tile t of one (batch, query head) and walks key tiles 0..t.
// Warp roles (384 threads):
//   warp 0      TMA producer: Q tile + scales once; K, V (columnwise, transposed) tiles + scales
//               through a 4-stage ring; the own-block token-normalised V tile once.
//   warp 1      allocates TMEM; lane 0 issues tcgen05.cp (scale factors, Q) and tcgen05.mma.
//   warp 2      decodes the token-normalised V tile to BF16 (exact) in the MMA operand layout.
//   warp 3      forwarder: turns each K/V stage's mbarrier completion into a named-barrier
//               generation for warp 1.
//   warps 4-11  softmax: each warp owns 16 query rows (TMEM 16x256b shape: a row's keys spread over
//               a quad of lanes, reductions are quad shuffles); then the epilogue, where warps 4+q
//               and 8+q store the two 64-column halves of rows 32q..32q+31.
// TMEM (512 columns): S[0] 0-127, S[1] 128-255, O 256-383, scale factors 384-411, Q 416-447 (the
// QK MMA reads Q from tensor memory and only K from shared memory).
// P (E4M3, 32 columns per term) is written over the S buffer it came from; the own-block BF16 P
// goes to the other S buffer.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "bsc_internal.h"
#include "ptx.cuh"

namespace bsc {

namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // keys per tile
constexpr int HD = 128;   // head dimension
constexpr int NST = 4;    // K/V shared-memory stages
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + BM * HD;              // NST stages, 128 keys x 128 d
constexpr uint32_t OFF_V = OFF_K + NST * BN * HD;        // NST stages, 128 d rows x 128 keys
constexpr uint32_t OFF_VT = OFF_V + NST * HD * BN;       // own-block V, BF16, 2 K-atoms of 16 KB
constexpr uint32_t OFF_VTN8 = OFF_VT + 2 * HD * BN;      // raw token-normalised bytes [key][d]
constexpr uint32_t OFF_SFQ = OFF_VTN8 + BN * HD;
constexpr uint32_t OFF_SFK = OFF_SFQ + 512;              // NST stages
constexpr uint32_t OFF_SFV = OFF_SFK + NST * 512;        // NST stages
constexpr uint32_t OFF_SFP = OFF_SFV + NST * 512;        // P scale blocks: term 0, term 1
constexpr uint32_t OFF_VTNSC = OFF_SFP + 2 * 512;        // 128 token amplitudes
constexpr uint32_t OFF_RED = OFF_VTNSC + 128;            // float [2 parity][2 halves][128 rows] maxima
constexpr uint32_t OFF_REDL = OFF_RED + 2 * 2 * 128 * 4; // float [l | m][128 rows]
constexpr uint32_t OFF_BAR = OFF_REDL + 2 * 128 * 4;
constexpr uint32_t NUM_BARS = 32;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;    // tmem slot, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;        // alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// A stage holds K_j and V_j with their scales: FULL[st] completes when the copies land, FREE[st]
// when PV_j (the last reader) completes; FREE also tells the softmax that PV_j is done.
enum Bar : uint32_t {
  B_Q_FULL = 0,
  B_FULL = 1,                    // + stage
  B_FREE = B_FULL + NST,         // + stage
  B_S_FULL = B_FREE + NST,       // + S buffer
  B_O_FULL = B_S_FULL + 2,
  B_VTN_FULL,
  B_VT_READY,
  B_DRAIN,
  B_INJECT,
  B_COUNT,
};
static_assert(B_COUNT <= NUM_BARS, "barrier slots");

// TMEM column map
constexpr uint32_t T_S0 = 0, T_S1 = 128, T_O = 256, T_SFQ = 384, T_SFK = 388, T_SFV = 396, T_SFP = 404,
                   T_Q = 416;   // Q bytes (128 rows x 128 B = 32 columns), the QK MMA's A operand

// Softmax weights are p' = 2^(x - m_used + P_SHIFT) with x - m_used <= RESCALE_LOG2, so
// p' < 2^8.8 = 445.7 < 448.  P scale bytes: term 0 holds p' (scale 2^-P_SHIFT), term 1 the
// residual * 16 (scale 2^-(P_SHIFT+4)).  P_SHIFT + RESCALE_LOG2 = 8.8 fixes the largest weight; a
// smaller shift lets the running maximum lag further behind the row's scores before O must be
// rescaled (each rescale stalls the warp on the previous P.V), at the cost of E4M3 underflow for
// weights more than 2^-(P_SHIFT + 9.5) below the running maximum.
constexpr float P_SHIFT = 6.0f;
constexpr float RESCALE_LOG2 = 2.8f;
constexpr uint8_t SFP_TERM0 = 127 - 6;
constexpr uint8_t SFP_TERM1 = 127 - 10;

// wait-site codes reported through the device status word
enum Site : int {
  W_PROD_FREE = 1, W_MMA_Q, W_FWD_KV, W_MMA_VT, W_MMA_INJECT,
  W_SM_S, W_SM_PV, W_SM_O, W_DEC_VTN,
};

__device__ __forceinline__ float pow2_e8m0(uint32_t sb) {
  return sb == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(sb << 23);   // 2^(sb-127), sb <= 254
}

// Named barrier for the two softmax warps that share a TMEM lane quarter.
// Hardware named barriers between the MMA warp and the warps it waits for.  Unlike an mbarrier
// wait, which returns only once the waiting thread's tcgen05 MMAs in flight have drained, a named
// barrier leaves the tensor pipe busy.  Every participant passes every generation of these
// barriers, also after an abort, so none of them can wait forever.
constexpr uint32_t NB_KV = 5;   // forwarder warp + MMA warp: K_j, V_j landed
constexpr uint32_t NB_P = 6;    // softmax warps + MMA warp: P_j written
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void pair_sync(int q) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
}

template <int P_TERMS, bool LEAKY>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](uint32_t i) { return sbase + OFF_BAR + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (a.S + BM - 1) / BM;   // the last tile may hold fewer rows (S is a multiple of 32)
  // heaviest tiles first; the query heads sharing a KV head are adjacent
  const int bh = blockIdx.x % (a.B * a.Hq);
  const int t = T - 1 - (int)(blockIdx.x / (a.B * a.Hq));
  const int hq = bh % a.Hq, b = bh / a.Hq;
  const int hk = hq / (a.Hq / a.Hkv);
  constexpr bool own_split = !LEAKY;

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_FREE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_S_FULL + s), 1);
    }
    mbar_init(bar(B_O_FULL), 1);
    mbar_init(bar(B_VTN_FULL), 1);
    mbar_init(bar(B_VT_READY), 32);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_INJECT), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_MISC, 512);
    tmem_relinquish();
  }
  // constant P scale blocks
  for (int i = threadIdx.x; i < 256; i += kThreads) {
    reinterpret_cast<uint32_t*>(smem + OFF_SFP)[i] = i < 128 ? SFP_TERM0 * 0x01010101u : SFP_TERM1 * 0x01010101u;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, a.dev_status, a.limit_ns};

  if (warp == 0) {
    // ======================= producer
    if (lane == 0) {
      prefetch_tensormap(&a.tm_q);
      prefetch_tensormap(&a.tm_k);
      prefetch_tensormap(&a.tm_v);
      const long long kv_plane = (long long)b * a.Hkv + hk;
      mbar_arrive_expect_tx(bar(B_Q_FULL), BM * HD + 512);
      tma_load_4d(sbase + OFF_Q, &a.tm_q, bar(B_Q_FULL), 0, hq, t * BM, b);
      bulk_load(sbase + OFF_SFQ, a.q_sc + (((long long)b * a.Hq + hq) * T + t) * 512, 512, bar(B_Q_FULL));
      if (own_split) {
        // the own-block tile of the token-normalised V, decoded early by warp 2
        prefetch_tensormap(&a.tm_vtn);
        // amplitudes of the tile's keys that exist (a multiple of 32); the decode zeroes the rest
        const uint32_t namp = (uint32_t)min(BN, a.S - t * BN);
        mbar_arrive_expect_tx(bar(B_VTN_FULL), BN * HD + namp);
        tma_load_4d(sbase + OFF_VTN8, &a.tm_vtn, bar(B_VTN_FULL), 0, hk, t * BN, b);
        bulk_load(sbase + OFF_VTNSC, a.vtn_sc + kv_plane * a.S + (long long)t * BN, namp, bar(B_VTN_FULL));
      }
      int nl[NST] = {};   // stage loads issued
      bool ok = true;
      for (int j = 0; j <= t && ok; ++j) {
        const int st = j % NST, n = j / NST;
        if (n > 0 && !(ok = mbar_wait(bar(B_FREE + st), (n - 1) & 1, ctl, W_PROD_FREE))) break;
        mbar_arrive_expect_tx(bar(B_FULL + st), 2 * BN * HD + 1024);
        tma_load_4d(sbase + OFF_K + st * BN * HD, &a.tm_k, bar(B_FULL + st), 0, hk, j * BN, b);
        bulk_load(sbase + OFF_SFK + st * 512, a.k_sc + (kv_plane * T + j) * 512, 512, bar(B_FULL + st));
        tma_load_2d(sbase + OFF_V + st * HD * BN, &a.tm_v, bar(B_FULL + st), j * BN, (int)(kv_plane * HD));
        bulk_load(sbase + OFF_SFV + st * 512, a.v_sc + (kv_plane * T + j) * 512, 512, bar(B_FULL + st));
        ++nl[st];
      }
      // drain: every copy this thread issued must land before the CTA may exit
      for (int st = 0; st < NST; ++st) {
        if (nl[st] > 0) mbar_wait_drain(bar(B_FULL + st), (nl[st] - 1) & 1, a.limit_ns);
      }
      mbar_wait_drain(bar(B_Q_FULL), 0, a.limit_ns);
      if (own_split) mbar_wait_drain(bar(B_VTN_FULL), 0, a.limit_ns);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (lane 0; the whole warp meets the named barriers)
    const uint32_t tS[2] = {tmem + T_S0, tmem + T_S1};
    const uint64_t dQ = desc_kmajor_sw128(sbase + OFF_Q), dK = desc_kmajor_sw128(sbase + OFF_K),
                   dV = desc_kmajor_sw128(sbase + OFF_V);   // descriptors: start address in 16-byte units
    const uint64_t dSFK = desc_sf_block(sbase + OFF_SFK), dSFV = desc_sf_block(sbase + OFF_SFV);
    const uint32_t tO = tmem + T_O;
    bool ok = true;
    if (lane == 0) {
      if (a.inject_stall) ok = mbar_wait(bar(B_INJECT), 0, ctl, W_MMA_INJECT);   // nothing arrives here
      ok = ok && mbar_wait(bar(B_Q_FULL), 0, ctl, W_MMA_Q);
      if (ok) {
        tc_fence_after();
        tc_cp_32x128b_warpx4(tmem + T_SFQ, desc_sf_block(sbase + OFF_SFQ));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // Q into TMEM, 32 bytes of each row per copy
          asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(tmem + T_Q + 8 * kk), "l"(dQ + 2 * kk)
                       : "memory");
        }
        tc_cp_32x128b_warpx4(tmem + T_SFP, desc_sf_block(sbase + OFF_SFP));
        tc_cp_32x128b_warpx4(tmem + T_SFP + 4, desc_sf_block(sbase + OFF_SFP + 512));
      }
    }
    // Per key tile j: S_j = Q K_j^T once stage j has landed; then O += P_{j-1} V_{j-1} once the
    // softmax has written P_{j-1} (the own block follows in the diagonal tile).  Everything one
    // thread issues executes in order, so S_{j+1} overwrites P_{j-1} only after PV_{j-1} read it.
    for (int jj = 0; jj <= t + 1; ++jj) {
      if (jj <= t) {
        named_sync(NB_KV, 64);
        if (lane == 0 && ok) {
          const int j = jj, st = j % NST, sb = j & 1;
          tc_fence_after();
          tc_cp_32x128b_warpx4(tmem + T_SFK + 4 * sb, dSFK + (uint64_t)(st * 32));
          tc_cp_32x128b_warpx4(tmem + T_SFV + 4 * sb, dSFV + (uint64_t)(st * 32));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_mxf8_ts(tS[sb], tmem + T_Q + 8 * kk,
                        dK + (uint64_t)(st * (BN * HD / 16) + 2 * kk), idesc_mxf8(BM, BN, kk, kk),
                        tmem + T_SFQ, tmem + T_SFK + 4 * sb, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(B_S_FULL + sb));
        }
      }
      if (jj >= 1) {
        named_sync(NB_P, 32 + kSoftmaxThreads);
        if (lane == 0 && ok) {
          const int j = jj - 1, st = j % NST, sb = j & 1;
          if (j == t && own_split) ok = mbar_wait(bar(B_VT_READY), 0, ctl, W_MMA_VT);
          if (ok) {
            tc_fence_after();
#pragma unroll
            for (int term = 0; term < P_TERMS; ++term) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                mma_mxf8_ts(tO, tS[sb] + term * 32 + kk * 8,
                            dV + (uint64_t)(st * (HD * BN / 16) + 2 * kk), idesc_mxf8(BM, HD, kk, kk),
                            tmem + T_SFP + 4 * term, tmem + T_SFV + 4 * sb, (j > 0 || term > 0 || kk > 0) ? 1u : 0u);
              }
            }
            if (j == t && own_split) {
#pragma unroll
              for (int term = 0; term < P_TERMS; ++term) {
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                  mma_f16_ts(tO, tS[sb ^ 1] + term * 64 + s * 8,
                             desc_kmajor_sw128(sbase + OFF_VT + (s >> 2) * (HD * 128) + (s & 3) * 32),
                             idesc_bf16(BM, HD), 1u);
                }
              }
            }
            tc_commit(bar(B_FREE + st));
          }
        }
      }
      __syncwarp();
    }
    if (lane == 0) {
      if (ok) tc_commit(bar(B_O_FULL));
      // drain every tcgen05 operation this thread issued before TMEM is released
      tc_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, a.limit_ns);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ======================= own-block V decode (32 threads)
    if (own_split) {
      const int u = lane;
      if (__all_sync(0xFFFFFFFFu, mbar_wait(bar(B_VTN_FULL), 0, ctl, W_DEC_VTN))) {
        const uint8_t* raw = smem + OFF_VTN8;
        const uint8_t* amp = smem + OFF_VTNSC;
        const int nkeys = min(BN, a.S - t * BN);   // keys past S: bytes zero-filled, no amplitude
        for (int part = 0; part < 4; ++part) {
          const int d = u + 32 * part;
          for (int kc = 0; kc < 16; ++kc) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              // slots 8kc + 2e + {0,1} carry keys k0, k0 + 1 (the order of the own-block BF16 P)
              const int k0 = 16 * (kc >> 1) + 8 * (e & 1) + 4 * (kc & 1) + 2 * (e >> 1);
              const uint16_t pair = (uint16_t)raw[k0 * HD + d] | ((uint16_t)raw[(k0 + 1) * HD + d] << 8);
              const uint32_t h2 = cvt_e4m3x2_to_f16x2(pair);
              const float v0 = k0 < nkeys ? __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * pow2_e8m0(amp[k0]) : 0.f;
              const float v1 = k0 + 1 < nkeys ? __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * pow2_e8m0(amp[k0 + 1]) : 0.f;
              w[e] = pack_bf16x2(v0, v1);
            }
            const uint32_t off = OFF_VT + (kc >> 3) * (HD * 128) + d * 128 + (((kc & 7) ^ (d & 7)) * 16);
            *reinterpret_cast<uint4*>(smem + off) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(bar(B_VT_READY));
    }
  } else if (warp == 3) {
    // ======================= forwarder: stage j has landed -> named barrier with the MMA warp
    for (int j = 0; j <= t; ++j) {
      (void)__all_sync(0xFFFFFFFFu, mbar_wait(bar(B_FULL + j % NST), (j / NST) & 1, ctl, W_FWD_KV));
      named_sync(NB_KV, 64);
    }
  } else {
    // ======================= softmax + epilogue (256 threads)
    // Warp w (4..11) owns the 16 query rows 32q + 16hf .. +15 of the tile (q = w % 4 is its TMEM
    // lane quarter, hf = (w - 4) / 4).  With the 16x256b TMEM shape, thread t holds rows
    // ra = base + t/4 and rb = ra + 8 for the keys 8k + 2(t%4) + {0,1}, k = 0..15: a row's 128
    // keys are spread over the four threads of a quad, so row reductions are quad shuffles and the
    // eight softmax warps run independently.  P is written in the same layout; inside each 32-key
    // block the MMA's K slot 8a + 2b + e carries key 8b + 2a + e (a 4x4 transpose of key pairs),
    // and the columnwise V bytes are stored in that key order, so P.V sums the same products.
    const int q = warp & 3;
    const int hf = (warp - 4) >> 2;
    const int qd = lane & 3;
    const int base = q * 32 + hf * 16;
    const int ra = base + (lane >> 2), rb = ra + 8;    // rows inside the tile
    const uint32_t lane_off = (uint32_t)base << 16;
    const float sl2 = a.scale_log2e;
    float* redl = reinterpret_cast<float*>(smem + OFF_REDL);   // [l | m][128 rows]
    // Exponentials are taken against m_a / m_b, running row maxima (log2 units) raised only when a
    // tile's maximum exceeds them by more than RESCALE_LOG2; O is rescaled then.  The weights
    // p' = 2^(x - m + P_SHIFT) stay below 2^(P_SHIFT + RESCALE_LOG2) < 448, inside the E4M3 range,
    // and every decision depends only on the row's own visible scores.
    float m_a = -INFINITY, m_b = -INFINITY;
    float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);   // partial row sums (this quad lane)
    bool ok = true;
    for (int j = 0; j <= t; ++j) {
      const int sb = j & 1;
      // one pass; a failed wait leaves it early (break) but the tile loop goes on to the barrier
      do {
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_S_FULL + sb), (j >> 1) & 1, ctl, W_SM_S));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tSb = tmem + (sb ? T_S1 : T_S0) + lane_off;
      float v[64];
      tmem_ld16x256_x16(tSb, v);
      tmem_ld_wait();
      const bool diag = (j == t);
      if (diag) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = 8 * k + 2 * qd + e;
            v[4 * k + e] = key > ra ? -INFINITY : v[4 * k + e];
            v[4 * k + 2 + e] = key > rb ? -INFINITY : v[4 * k + 2 + e];
          }
        }
      }
      // row maxima: 32 values per row in this lane (k = 0..15), then across the quad
      float xa0 = fmax3(v[0], v[1], v[4]), xa1 = fmax3(v[5], v[8], v[9]);
      float xb0 = fmax3(v[2], v[3], v[6]), xb1 = fmax3(v[7], v[10], v[11]);
#pragma unroll
      for (int k = 3; k < 15; k += 2) {
        xa0 = fmax3(xa0, v[4 * k], v[4 * k + 1]);
        xa1 = fmax3(xa1, v[4 * k + 4], v[4 * k + 5]);
        xb0 = fmax3(xb0, v[4 * k + 2], v[4 * k + 3]);
        xb1 = fmax3(xb1, v[4 * k + 6], v[4 * k + 7]);
      }
      float mta = fmax3(xa0, xa1, fmaxf(v[60], v[61])), mtb = fmax3(xb0, xb1, fmaxf(v[62], v[63]));
      mta = fmaxf(mta, __shfl_xor_sync(0xFFFFFFFFu, mta, 1));
      mtb = fmaxf(mtb, __shfl_xor_sync(0xFFFFFFFFu, mtb, 1));
      mta = fmaxf(mta, __shfl_xor_sync(0xFFFFFFFFu, mta, 2)) * sl2;
      mtb = fmaxf(mtb, __shfl_xor_sync(0xFFFFFFFFu, mtb, 2)) * sl2;
      const bool need_a = mta > m_a + RESCALE_LOG2, need_b = mtb > m_b + RESCALE_LOG2;   // true at j = 0
      const float mna = need_a ? mta : m_a, mnb = need_b ? mtb : m_b;
      const bool resc = (need_a || need_b) && (j > 0);
      bool pv_waited = false;
      if (__any_sync(0xFFFFFFFFu, resc)) {
        // rescale this warp's O rows (factor 1 for rows that keep their max): needs PV_{j-1} done
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_FREE + (j - 1) % NST), ((j - 1) / NST) & 1, ctl, W_SM_PV));
        if (!ok) break;
        pv_waited = true;
        tc_fence_after();
        const float alpha_a = (need_a && j > 0) ? ex2_approx(m_a - mna) : 1.0f;
        const float alpha_b = (need_b && j > 0) ? ex2_approx(m_b - mnb) : 1.0f;
        const uint32_t tOb = tmem + T_O + lane_off;
        uint32_t o[64];
        tmem_ld16x256_x16u(tOb, o);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          o[4 * k + 0] = __float_as_uint(__uint_as_float(o[4 * k + 0]) * alpha_a);
          o[4 * k + 1] = __float_as_uint(__uint_as_float(o[4 * k + 1]) * alpha_a);
          o[4 * k + 2] = __float_as_uint(__uint_as_float(o[4 * k + 2]) * alpha_b);
          o[4 * k + 3] = __float_as_uint(__uint_as_float(o[4 * k + 3]) * alpha_b);
        }
        tmem_st16x256_x16(tOb, o);
        la.x *= alpha_a; la.y *= alpha_a;
        lb.x *= alpha_b; lb.y *= alpha_b;
      }
      m_a = mna;
      m_b = mnb;
      // p' = 2^(s * scale*log2(e) - m + P_SHIFT)
      const float2 mul2 = make_float2(sl2, sl2);
      const float2 adda = make_float2(P_SHIFT - m_a, P_SHIFT - m_a), addb = make_float2(P_SHIFT - m_b, P_SHIFT - m_b);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 xa = __ffma2_rn(make_float2(v[4 * k], v[4 * k + 1]), mul2, adda);
        const float2 xb = __ffma2_rn(make_float2(v[4 * k + 2], v[4 * k + 3]), mul2, addb);
        v[4 * k] = ex2_approx(xa.x);
        v[4 * k + 1] = ex2_approx(xa.y);
        v[4 * k + 2] = ex2_approx(xb.x);
        v[4 * k + 3] = ex2_approx(xb.y);
        la = __fadd2_rn(la, make_float2(v[4 * k], v[4 * k + 1]));
        lb = __fadd2_rn(lb, make_float2(v[4 * k + 2], v[4 * k + 3]));
      }
      // E4M3 P (scale 2^-P_SHIFT; a second term holds the residual at 2^-4 of that) over this S
      // buffer: block kb's columns 8kb + 2qd and 8kb + 2qd + 1 carry keys {8(4kb) + 2qd + e,
      // 8(4kb+1) + 2qd + e} and {8(4kb+2) ..., 8(4kb+3) ...}.  In the diagonal tile the blocks after
      // the own block are masked to 0 already; the own block's words are cleared below (the leaky
      // control keeps the own block on this path instead).
      uint32_t w0[16], w1[16];
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int k0 = 4 * kb + 2 * c2;   // keys 8k0 + 2qd + e and 8(k0+1) + 2qd + e
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const float p0 = v[4 * k0 + 2 * rr], p1 = v[4 * k0 + 2 * rr + 1];
            const float p2 = v[4 * k0 + 4 + 2 * rr], p3 = v[4 * k0 + 4 + 2 * rr + 1];
            const uint16_t h01 = cvt_e4m3x2(p0, p1), h23 = cvt_e4m3x2(p2, p3);
            w0[4 * kb + 2 * rr + c2] = (uint32_t)h01 | ((uint32_t)h23 << 16);
            if (P_TERMS > 1) {
              const uint32_t f01 = cvt_e4m3x2_to_f16x2(h01), f23 = cvt_e4m3x2_to_f16x2(h23);
              const float d0 = p0 - __half2float(__ushort_as_half((unsigned short)(f01 & 0xFFFFu)));
              const float d1 = p1 - __half2float(__ushort_as_half((unsigned short)(f01 >> 16)));
              const float d2 = p2 - __half2float(__ushort_as_half((unsigned short)(f23 & 0xFFFFu)));
              const float d3 = p3 - __half2float(__ushort_as_half((unsigned short)(f23 >> 16)));
              w1[4 * kb + 2 * rr + c2] =
                  (uint32_t)cvt_e4m3x2(d0 * 16.f, d1 * 16.f) | ((uint32_t)cvt_e4m3x2(d2 * 16.f, d3 * 16.f) << 16);
            }
          }
        }
      }
      if (diag && !LEAKY) {
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          if (kb == q) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              w0[4 * kb + i] = 0u;
              w1[4 * kb + i] = 0u;
            }
          }
        }
      }
      tmem_st16x256_x4(tSb, w0);
      if (P_TERMS > 1) tmem_st16x256_x4(tSb + 32, w1);
      if (diag && !LEAKY) {
        // own block (keys of sub-block q, key <= row) as BF16 P (P_TERMS terms) into the other S
        // buffer once PV_{t-1}, its last reader, is done.  16-key group g16: column 8g16 + 2qd
        // carries keys 16g16 + 2qd + e, column 8g16 + 2qd + 1 keys 16g16 + 8 + 2qd + e (the decoded
        // V tile uses the same key order).
        if (t > 0 && !pv_waited) {
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_FREE + (t - 1) % NST), ((t - 1) / NST) & 1, ctl, W_SM_PV));
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t tPo = tmem + (sb ? T_S0 : T_S1) + lane_off;
        const float unshift = 1.0f / (float)(1 << (int)P_SHIFT);
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int g16 = 0; g16 < 8; ++g16) {
          const bool own = (g16 >> 1) == q;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int k = 2 * g16 + m;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const float p0 = own ? v[4 * k + 2 * rr] * unshift : 0.f;
              const float p1 = own ? v[4 * k + 2 * rr + 1] * unshift : 0.f;
              const uint32_t hh = pack_bf16x2(p0, p1);
              hi[4 * g16 + 2 * rr + m] = hh;
              lo[4 * g16 + 2 * rr + m] =
                  pack_bf16x2(p0 - __uint_as_float(hh << 16), p1 - __uint_as_float(hh & 0xFFFF0000u));
            }
          }
        }
        tmem_st16x256_x8(tPo, hi);
        if (P_TERMS > 1) tmem_st16x256_x8(tPo + 64, lo);
      }
      } while (false);
      tmem_st_wait();
      tc_fence_before();
      named_sync(NB_P, 32 + kSoftmaxThreads);   // P_j written (or this warp gave up)
    }
    // ---- epilogue: row sums across the quad, then O / l -> BF16 and the LSE, with the 32x32b
    // shape: warp 4+q stores columns 0-63 and warp 8+q columns 64-127 of rows 32q..32q+31
    float sa = la.x + la.y, sbm = lb.x + lb.y;
    sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 1);
    sbm += __shfl_xor_sync(0xFFFFFFFFu, sbm, 1);
    sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 2);
    sbm += __shfl_xor_sync(0xFFFFFFFFu, sbm, 2);
    if (qd == 0) {
      redl[ra] = sa;
      redl[rb] = sbm;
      redl[128 + ra] = m_a;
      redl[128 + rb] = m_b;
    }
    pair_sync(q);
    if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_O_FULL), 0, ctl, W_SM_O));
    if (ok) {
      tc_fence_after();
      const int h = hf;
      const int r = q * 32 + lane;        // row inside the tile
      const int i = t * BM + r;           // query token
      const float l = redl[r], m_fin = redl[128 + r];
      const float inv_l = (float)(1 << (int)P_SHIFT) / l;
      const long long row = a.layout == 0 ? ((long long)b * a.S + i) * a.Hq + hq
                                          : ((long long)i * a.B + b) * a.Hq + hq;
      const uint32_t tOb = tmem + T_O + ((uint32_t)(q * 32) << 16) + 64 * h;
      float o[2][32];
      tmem_ld32f(tOb, o[0]);
      tmem_ld32f(tOb + 32, o[1]);
      tmem_ld_wait();
      const bool row_ok = i < a.S;   // rows past S hold no token
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[c][e] *= inv_l;
      }
      if (a.o != nullptr) {
        uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) + row * HD + 64 * h);
#pragma unroll
        for (int e8 = 0; e8 < 8; ++e8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = e8 * 8 + 2 * e;
            w[e] = pack_bf16x2(o[k >> 5][k & 31], o[(k + 1) >> 5][(k + 1) & 31]);
          }
          if (row_ok) orow[e8] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if (a.o8 != nullptr) {
        // MXFP8 O: this thread's 64 columns are the 32-element blocks 2h and 2h + 1 of row r, so each
        // block maximum is thread-local.  The maximum is taken on |bit patterns| (NaN above Inf above
        // every finite value); scales go to row r's word of the tile's row atom.
        uint8_t* atom = a.o_sc + (((long long)b * a.Hq + hq) * T + t) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t mb = 0;
#pragma unroll
          for (int e = 0; e < 32; ++e) mb = max(mb, __float_as_uint(o[c][e]) & 0x7FFFFFFFu);
          float inv;
          const uint32_t sbyte = e8m0_from_amax(__uint_as_float(mb), inv);
          uint32_t wq[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t lo = cvt_e4m3x2(o[c][4 * k] * inv, o[c][4 * k + 1] * inv);
            const uint32_t hi = cvt_e4m3x2(o[c][4 * k + 2] * inv, o[c][4 * k + 3] * inv);
            wq[k] = sbyte == 0xFFu ? 0x7F7F7F7Fu : (lo | (hi << 16));
          }
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(a.o8 + row * HD + 64 * h + 32 * c);
            dst[0] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
            dst[1] = make_uint4(wq[4], wq[5], wq[6], wq[7]);
          }
          atom[2 * h + c] = row_ok ? (uint8_t)sbyte : (uint8_t)0;
        }
      }
      if (h == 0 && i < a.S) {
        const float ln2 = 0.69314718055994531f;
        a.lse[((long long)b * a.Hq + hq) * a.S + i] = (m_fin + lg2_approx(l) - P_SHIFT) * ln2;
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int P_TERMS, bool LEAKY>
cudaError_t launch_variant(const AttnArgs& args, cudaStream_t st) {
  static bool attr_set = false;   // the attribute is per function and per process
  auto kern = attn_fwd_kernel<P_TERMS, LEAKY>;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long ctas = (long long)args.B * args.Hq * ((args.S + BM - 1) / BM);
  kern<<<(unsigned)ctas, kThreads, SMEM_BYTES, st>>>(args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnArgs& args, cudaStream_t st) {
  if (args.p_terms == 2) return args.leaky ? launch_variant<2, true>(args, st) : launch_variant<2, false>(args, st);
  return args.leaky ? launch_variant<1, true>(args, st) : launch_variant<1, false>(args, st);
}

}  // namespace bsc
