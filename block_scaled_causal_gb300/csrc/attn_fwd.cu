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
// Work unit: one CTA takes two 128-row query tiles ("slots") that read the same KV head and walks
// the key tiles 0..t0 once, each K/V tile serving both slots.  Slot 0 is the tile with the larger
// (or equal) index t0, slot 1 has t1 = t0 or t0 - 1 (query heads of a GQA group at the same tile,
// or neighbouring tiles of one head).  The MMA warp alternates between the slots, so that one
// slot's softmax runs while the tensor cores work on the other slot.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: both query tiles with their compact scales; K and V (columnwise,
//               transposed) tiles with their compact scales through a 3-stage ring.
//   warp 1      allocates TMEM; the warp meets the named barriers, its lane 0 issues tcgen05.cp
//               (scale factors) and tcgen05.mma.
//   warp 2      decodes the own-block tiles of the token-normalised V to BF16 (exact).
//   warp 3      forwarder: waits for each K/V stage, permutes its compact scales into the
//               tensor-core scale-factor atoms and releases the stage to the MMA warp through a
//               named barrier.
//   warps 4-7   softmax of slot 0, warps 8-11 softmax of slot 1: one query row per thread (TMEM
//               32x32b shape), then that slot's epilogue.
// TMEM (512 columns): S of slot 0 (0-127), S of slot 1 (128-255), O of slot 0 (256-383), O of
// slot 1 (384-511).  Scale factors live in S columns that are dead when they are needed: the P.V
// scales in the slot's own S after its softmax has written P, the next QK scales in the other
// slot's S after that slot's softmax has loaded its scores.
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
constexpr int NST = 3;    // K/V shared-memory stages
constexpr int kThreads = 384;
constexpr uint32_t kSlotThreads = 128;   // softmax threads per slot

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t TILE8 = BM * HD;                      // one 128 x 128 E4M3 tile
constexpr uint32_t VT_BYTES = 2 * BN * HD;               // one BF16 own-block V tile
constexpr uint32_t OFF_Q = 0;                            // 2 slots
constexpr uint32_t OFF_K = OFF_Q + 2 * TILE8;            // NST stages, 128 keys x 128 d
constexpr uint32_t OFF_V = OFF_K + NST * TILE8;          // NST stages, 128 d rows x 128 keys
constexpr uint32_t OFF_VT = OFF_V + NST * TILE8;         // 2 buffers: own-block V, BF16 [key][d]
constexpr uint32_t OFF_QSC = OFF_VT + 2 * VT_BYTES;      // compact Q scales, 2 slots x 512
constexpr uint32_t OFF_QATOM = OFF_QSC + 2 * 512;        // Q scale atoms, 2 slots
constexpr uint32_t OFF_KSC = OFF_QATOM + 2 * 512;        // compact K scales, NST stages
constexpr uint32_t OFF_VSC = OFF_KSC + NST * 512;        // compact V scales, NST stages
constexpr uint32_t OFF_KATOM = OFF_VSC + NST * 512;      // K scale atoms, NST stages
constexpr uint32_t OFF_VATOM = OFF_KATOM + NST * 512;    // V scale atoms, NST stages
constexpr uint32_t OFF_PATOM = OFF_VATOM + NST * 512;    // P scale atoms, 2 slots
constexpr uint32_t OFF_BAR = OFF_PATOM + 2 * 512;
constexpr uint32_t NUM_BARS = 24;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;    // tmem slot, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;        // alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// mbarriers.  FULL[st] completes when stage st's copies land; FREE[st] when the last MMA reading
// the stage has completed.  S_FULL[x]: slot x's scores are in TMEM (and every earlier MMA of the
// issuing thread, in particular slot x's previous P.V, has completed).  O_FULL[x]: slot x's O is
// final.  VT_READY[b]: own-block V buffer b is decoded.
enum Bar : uint32_t {
  B_Q_FULL = 0,
  B_FULL = 1,                    // + stage
  B_FREE = B_FULL + NST,         // + stage
  B_S_FULL = B_FREE + NST,       // + slot
  B_O_FULL = B_S_FULL + 2,       // + slot
  B_VT_READY = B_O_FULL + 2,     // + buffer
  B_DRAIN = B_VT_READY + 2,
  B_INJECT,
  B_COUNT,
};
static_assert(B_COUNT <= NUM_BARS, "barrier slots");

// TMEM columns
constexpr uint32_t T_S0 = 0, T_O0 = 256;   // slot x: S at T_S0 + 128x, O at T_O0 + 128x
// Column offsets inside a slot's S region once its softmax has loaded the scores.
//   ordinary tile:            P term 0 [0,32), P term 1 [32,64), P.V scales [64,72),
//                             the other slot's next QK scales [96,104)
//   own-block diagonal tile:  P term 0 [0,24) (key blocks 0-2), P.V scales [24,32),
//                             P term 1 [32,56), a deferred QK's scales [56,64),
//                             own-block BF16 P [64,128)
// Each scale pair is (A scales, B scales) in 4 + 4 columns.
constexpr uint32_t C_P1 = 32, C_OWNP = 64;
constexpr uint32_t C_SF_PV = 64, C_SF_PV_DIAG = 24, C_SF_QK = 96, C_SF_QK_DIAG = 56;

// The running row maximum m (log2 units) is raised only when a tile's maximum exceeds it by more
// than RESCALE_LOG2; O and l are then rescaled.  P is stored relative to a power-of-two scale
// chosen per row and 32-key block (see the softmax), so the lag costs no E4M3 range.
constexpr float RESCALE_LOG2 = 8.0f;

// wait-site codes reported through the device status word
enum Site : int {
  W_PROD_FREE = 1, W_MMA_Q, W_FWD_KV, W_MMA_VT, W_MMA_INJECT,
  W_SM_S, W_SM_PV, W_SM_O, W_DEC_VTN, W_FWD_Q,
};

// Named barriers (ID 0 is __syncthreads).  The MMA warp waits on these only: an mbarrier wait in
// the thread that issues tcgen05.mma returns only once that thread's MMAs in flight have drained,
// a hardware named barrier does not.  Producers arrive without blocking when their next arrival
// cannot overtake the MMA warp (it depends on an MMA the warp issues after this barrier), and
// block (bar.sync) otherwise, so that no barrier ever sees arrivals of two generations.
constexpr uint32_t NB_KV = 1;   // forwarder + MMA warp: a K/V stage (and at first, Q) is ready
constexpr uint32_t NB_P = 2;    // + slot: slot's softmax + MMA warp: P and its scales written
constexpr uint32_t NB_SL = 4;   // + slot: slot's softmax + MMA warp: scores loaded, S is free
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t count) {
  asm volatile("barrier.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float pow2_e8m0(uint32_t sb) {
  return sb == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(sb << 23);   // 2^(sb-127), sb <= 254
}

// The two query tiles of this CTA.  Tiles of one KV group are listed by descending tile index,
// query heads ascending within a tile index, and paired in that order; CTAs go pair-major with
// the groups interleaved, so the heaviest pairs run first and CTAs of one group that run at the
// same time read the same K/V tiles.
struct Unit {
  int b, hk, t0, t1, hq0, hq1;
  bool has1;
};
__device__ __forceinline__ Unit decode_unit(const AttnArgs& a, int T) {
  const int g = a.Hq / a.Hkv;
  const int ngroups = a.B * a.Hkv;
  const int grp = (int)(blockIdx.x % (unsigned)ngroups), p = (int)(blockIdx.x / (unsigned)ngroups);
  Unit u;
  u.b = grp / a.Hkv;
  u.hk = grp % a.Hkv;
  const int i0 = 2 * p, i1 = 2 * p + 1;
  u.has1 = i1 < T * g;
  u.t0 = T - 1 - i0 / g;
  u.hq0 = u.hk * g + i0 % g;
  u.t1 = u.has1 ? T - 1 - i1 / g : -1;
  u.hq1 = u.has1 ? u.hk * g + i1 % g : 0;
  return u;
}

// Compact rowwise scales (one 32-bit word per row, byte c for the 32-element block c) -> the
// tensor-core scale-factor atom: row m's word at (m % 32) * 16 + (m / 32) * 4.  Rows at or past
// `nrows` get 0.  One warp; lane l writes the atom's 16-byte line l.
__device__ __forceinline__ void rows_to_atom(const uint8_t* compact, uint8_t* atom, int nrows, int lane) {
  const uint32_t* src = reinterpret_cast<const uint32_t*>(compact);
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] = lane + 32 * k < nrows ? src[lane + 32 * k] : 0u;
  *reinterpret_cast<uint4*>(atom + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
}
// Compact columnwise V scales of one 128-token tile (block kb's 128 bytes, one per d, at
// kb * 128 + d) -> the atom: d's word at (d % 32) * 16 + (d / 32) * 4, byte kb.  Blocks at or
// past `nblk` get 0.  Lane l handles d = 4l .. 4l + 3 (a 4 x 4 byte transpose).
__device__ __forceinline__ void cols_to_atom(const uint8_t* compact, uint8_t* atom, int nblk, int lane) {
  const uint32_t* src = reinterpret_cast<const uint32_t*>(compact);
  uint32_t w[4];
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) w[kb] = kb < nblk ? src[kb * 32 + lane] : 0u;
  const uint32_t t0 = __byte_perm(w[0], w[1], 0x5140), t1 = __byte_perm(w[2], w[3], 0x5140);
  const uint32_t t2 = __byte_perm(w[0], w[1], 0x7362), t3 = __byte_perm(w[2], w[3], 0x7362);
  const uint32_t o[4] = {__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632), __byte_perm(t2, t3, 0x5410),
                         __byte_perm(t2, t3, 0x7632)};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int d = 4 * lane + e;
    *reinterpret_cast<uint32_t*>(atom + (d & 31) * 16 + (d >> 5) * 4) = o[e];
  }
}

// 2^e for an integer e in [-127, 127], exactly.
__device__ __forceinline__ float exp2i(int e) {
  return e >= -126 ? __int_as_float((e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Packed f32 pair -> f16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// f16x2 -> packed E4M3x2 (round to nearest even, saturating); low half -> low byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2_f16x2(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// TMEM loads/stores of one thread's row (32x32b shape) from/to register arrays given by pointer.
__device__ __forceinline__ void tld32(uint32_t taddr, float* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]),
        "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15]),
        "=f"(r[16]), "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]),
        "=f"(r[24]), "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]), "=f"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tst16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tst8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// Eight E4M3 bytes (one uint2) * scale -> eight BF16 (one uint4); exact for in-range values.
__device__ __forceinline__ uint4 decode8(uint2 bytes, float scale) {
  const uint32_t bw[2] = {bytes.x, bytes.y};
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t h2 = cvt_e4m3x2_to_f16x2((uint16_t)(bw[e >> 1] >> (16 * (e & 1))));
    w[e] = pack_bf16x2(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * scale,
                       __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * scale);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int P_TERMS, bool LEAKY>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](uint32_t i) { return sbase + OFF_BAR + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  constexpr bool OWN = !LEAKY;   // the own block goes through the token-normalised V

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (a.S + BM - 1) / BM;   // the last tile may hold fewer rows (S is a multiple of 32)
  const Unit u = decode_unit(a, T);
  const int b = u.b, hk = u.hk, t0 = u.t0, t1 = u.t1;
  const bool has1 = u.has1;
  const long long kv_plane = (long long)b * a.Hkv + hk;
  // own-block V buffers: slot 1's diagonal tile first (it comes first), then slot 0's if different
  const int nvt = (OWN ? ((has1 && t1 != t0) ? 2 : 1) : 0);
  const int vt_buf0 = (has1 && t1 != t0) ? 1 : 0;   // slot 0's buffer; slot 1 uses buffer 0

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_FREE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_S_FULL + s), 1);
      mbar_init(bar(B_O_FULL + s), 1);
      mbar_init(bar(B_VT_READY + s), 1);
    }
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_INJECT), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_MISC, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, a.dev_status, a.limit_ns};
  // Registers: the launch gives 168 per thread (384 x 168 = 64512).  The four control warps keep
  // 112, the eight softmax warps get 192: 128 x 112 + 256 x 192 = 63488.
  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
  if (warp == 0) {
    // ======================= producer
    if (lane == 0) {
      prefetch_tensormap(&a.tm_q);
      prefetch_tensormap(&a.tm_k);
      prefetch_tensormap(&a.tm_v);
      const int nr0 = min(BM, a.S - t0 * BM), nr1 = has1 ? min(BM, a.S - t1 * BM) : 0;
      mbar_arrive_expect_tx(bar(B_Q_FULL), (has1 ? 2 : 1) * TILE8 + 4u * (uint32_t)(nr0 + nr1));
      tma_load_4d(sbase + OFF_Q, &a.tm_q, bar(B_Q_FULL), 0, u.hq0, t0 * BM, b);
      bulk_load(sbase + OFF_QSC, a.q_sc + (((long long)b * a.Hq + u.hq0) * a.S + (long long)t0 * BM) * 4,
                4u * (uint32_t)nr0, bar(B_Q_FULL));
      if (has1) {
        tma_load_4d(sbase + OFF_Q + TILE8, &a.tm_q, bar(B_Q_FULL), 0, u.hq1, t1 * BM, b);
        bulk_load(sbase + OFF_QSC + 512, a.q_sc + (((long long)b * a.Hq + u.hq1) * a.S + (long long)t1 * BM) * 4,
                  4u * (uint32_t)nr1, bar(B_Q_FULL));
      }
      int nl[NST] = {};   // stage loads issued
      bool ok = true;
      for (int j = 0; j <= t0 && ok; ++j) {
        const int st = j % NST, n = j / NST;
        if (n > 0 && !(ok = mbar_wait(bar(B_FREE + st), (n - 1) & 1, ctl, W_PROD_FREE))) break;
        const int nk = min(BN, a.S - j * BN);
        mbar_arrive_expect_tx(bar(B_FULL + st), 2 * TILE8 + 4u * (uint32_t)nk + 4u * (uint32_t)nk);
        tma_load_4d(sbase + OFF_K + st * TILE8, &a.tm_k, bar(B_FULL + st), 0, hk, j * BN, b);
        bulk_load(sbase + OFF_KSC + st * 512, a.k_sc + (kv_plane * a.S + (long long)j * BN) * 4, 4u * (uint32_t)nk,
                  bar(B_FULL + st));
        tma_load_2d(sbase + OFF_V + st * TILE8, &a.tm_v, bar(B_FULL + st), j * BN, (int)(kv_plane * HD));
        // V scales: nk / 32 blocks of 128 bytes
        bulk_load(sbase + OFF_VSC + st * 512, a.v_sc + (kv_plane * (a.S / 32) + (long long)j * 4) * 128,
                  4u * (uint32_t)nk, bar(B_FULL + st));
        ++nl[st];
      }
      // drain: every copy this thread issued must land before the CTA may exit
      for (int st = 0; st < NST; ++st) {
        if (nl[st] > 0) mbar_wait_drain(bar(B_FULL + st), (nl[st] - 1) & 1, a.limit_ns);
      }
      mbar_wait_drain(bar(B_Q_FULL), 0, a.limit_ns);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (lane 0; the whole warp meets the named barriers)
    const uint32_t tS[2] = {tmem + T_S0, tmem + T_S0 + 128};
    const uint32_t tO[2] = {tmem + T_O0, tmem + T_O0 + 128};
    const uint64_t dQ = desc_kmajor_sw128(sbase + OFF_Q), dK = desc_kmajor_sw128(sbase + OFF_K),
                   dV = desc_kmajor_sw128(sbase + OFF_V);   // descriptors: start address in 16-byte units
    const int tx[2] = {t0, t1};
    bool ok = true;
    if (lane == 0 && a.inject_stall) ok = mbar_wait(bar(B_INJECT), 0, ctl, W_MMA_INJECT);   // nothing arrives here
    // S_x = Q_x K_j^T with the Q and K scale atoms copied to columns sfc, sfc + 4
    auto issue_qk = [&](int x, int j, uint32_t sfc) {
      const int st = j % NST;
      tc_cp_32x128b_warpx4(sfc, desc_sf_block(sbase + OFF_QATOM + x * 512));
      tc_cp_32x128b_warpx4(sfc + 4, desc_sf_block(sbase + OFF_KATOM + st * 512));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_mxf8_ss(tS[x], dQ + (uint64_t)(x * (TILE8 / 16) + 2 * kk), dK + (uint64_t)(st * (TILE8 / 16) + 2 * kk),
                    idesc_mxf8(BM, BN, kk, kk), sfc, sfc + 4, kk > 0 ? 1u : 0u);
      }
      tc_commit(bar(B_S_FULL + x));
    };
    // O_x += P_x V_j (completed blocks, E4M3), then in the diagonal tile the own block (BF16)
    auto issue_pv = [&](int x, int j, bool own) {
      const int st = j % NST;
      const uint32_t sfc = tS[x] + (own ? C_SF_PV_DIAG : C_SF_PV);
      tc_cp_32x128b_warpx4(sfc, desc_sf_block(sbase + OFF_PATOM + x * 512));
      tc_cp_32x128b_warpx4(sfc + 4, desc_sf_block(sbase + OFF_VATOM + st * 512));
      const int nkk = own ? 3 : 4;   // key block 3 of a diagonal tile is never a completed block
#pragma unroll
      for (int term = 0; term < P_TERMS; ++term) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if (kk < nkk) {
            mma_mxf8_ts(tO[x], tS[x] + term * C_P1 + kk * 8, dV + (uint64_t)(st * (TILE8 / 16) + 2 * kk),
                        idesc_mxf8(BM, HD, kk, kk), sfc, sfc + 4, (j > 0 || term > 0 || kk > 0) ? 1u : 0u);
          }
        }
      }
      if (own) {
        const int buf = x == 1 ? 0 : vt_buf0;
        ok = mbar_wait(bar(B_VT_READY + buf), 0, ctl, W_MMA_VT);
        if (ok) {
          tc_fence_after();
          const uint32_t vt = sbase + OFF_VT + buf * VT_BYTES;
#pragma unroll
          for (int s = 0; s < 8; ++s) {   // B is [key][d]: MN-major, 16 keys = 2048 bytes per step
            mma_f16_ts(tO[x], tS[x] + C_OWNP + 8 * s, smem_desc(vt + s * 2048, 16384, 1024, 2),
                       idesc_bf16(BM, HD) | (1u << 16), 1u);
          }
        }
      }
      if (j == tx[x]) tc_commit(bar(B_O_FULL + x));
    };

    named_sync(NB_KV, 64);   // Q tiles, K/V tile 0
    if (lane == 0 && ok) {
      tc_fence_after();
      issue_qk(0, 0, tO[0]);   // O is first written by the slot's first P.V, after this QK
      if (has1) issue_qk(1, 0, tO[1]);
    }
    bool defer_qk1 = false;   // slot 1's QK of tile j waits for slot 0's own-block P.V of tile j
    for (int j = 0; j <= t0; ++j) {
      const bool act1 = has1 && j <= t1;
      const bool own0 = OWN && j == t0, own1 = OWN && act1 && j == t1;
      // ---- slot 0
      named_sync(NB_P + 0, 32 + kSlotThreads);
      if (lane == 0 && ok) {
        tc_fence_after();
        issue_pv(0, j, own0);
        if (defer_qk1 && ok) issue_qk(1, j, tS[0] + C_SF_QK_DIAG);
      }
      defer_qk1 = false;
      bool defer_qk0 = false;
      if (j < t0) {
        named_sync(NB_KV, 64);   // K/V tile j + 1
        if (own1) {
          defer_qk0 = true;   // slot 1's S holds its own-block P: no free columns until its P.V
        } else {
          if (act1) named_sync(NB_SL + 1, 32 + kSlotThreads);
          if (lane == 0 && ok) {
            tc_fence_after();
            issue_qk(0, j + 1, tS[1] + C_SF_QK);
          }
        }
      }
      // ---- slot 1
      if (act1) {
        named_sync(NB_P + 1, 32 + kSlotThreads);
        if (lane == 0 && ok) {
          tc_fence_after();
          issue_pv(1, j, own1);
          if (defer_qk0 && ok) issue_qk(0, j + 1, tS[1] + C_SF_QK_DIAG);
        }
        if (j < t1) {
          if (OWN && j + 1 == t0) {
            defer_qk1 = true;   // slot 0's next tile is its own-block diagonal tile
          } else {
            named_sync(NB_SL + 0, 32 + kSlotThreads);
            if (lane == 0 && ok) {
              tc_fence_after();
              issue_qk(1, j + 1, tS[0] + C_SF_QK);
            }
          }
        }
      }
      if (lane == 0 && ok) tc_commit(bar(B_FREE + j % NST));
      __syncwarp();
    }
    if (lane == 0) {
      // drain every tcgen05 operation this thread issued before TMEM is released
      tc_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, a.limit_ns);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ======================= own-block V decode (32 threads): token-normalised bytes [key][d] from
    // global memory, times the key's amplitude, to BF16 [key][d] in two 64-column blocks with the
    // 128-byte swizzle (the MN-major B operand of the own-block MMA).  Keys past S become 0.
    for (int buf = 0; buf < nvt; ++buf) {
      const int t = (buf == 0 && has1) ? t1 : t0;
      const int nkeys = min(BN, a.S - t * BN);
      uint8_t* dst = smem + OFF_VT + buf * VT_BYTES;
      for (int it = 0; it < 8; ++it) {   // 64 eight-element units per lane, 8 loads in flight
        uint2 raw[8];
        float sc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int unit = lane + 32 * (8 * it + k), key = unit >> 4, d0 = (unit & 15) * 8;
          const int tok = t * BN + key;
          raw[k] = make_uint2(0u, 0u);
          sc[k] = 0.f;
          if (key < nkeys) {
            const long long row = a.layout == 0 ? ((long long)b * a.S + tok) * a.Hkv + hk
                                                : ((long long)tok * a.B + b) * a.Hkv + hk;
            raw[k] = __ldg(reinterpret_cast<const uint2*>(a.vtn + row * HD + d0));
            sc[k] = pow2_e8m0(__ldg(a.vtn_sc + kv_plane * a.S + tok));
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int unit = lane + 32 * (8 * it + k), key = unit >> 4, d0 = (unit & 15) * 8;
          const uint32_t off = (uint32_t)(d0 >> 6) * 16384u + (uint32_t)key * 128u +
                               ((((uint32_t)(d0 & 63) >> 3) ^ ((uint32_t)key & 7u)) << 4);
          *reinterpret_cast<uint4*>(dst + off) = decode8(raw[k], sc[k]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_VT_READY + buf));
    }
  } else if (warp == 3) {
    // ======================= forwarder: scale atoms, then stage j -> named barrier with the MMA warp
    bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_Q_FULL), 0, ctl, W_FWD_Q));
    if (ok) {
      rows_to_atom(smem + OFF_QSC, smem + OFF_QATOM, min(BM, a.S - t0 * BM), lane);
      if (has1) rows_to_atom(smem + OFF_QSC + 512, smem + OFF_QATOM + 512, min(BM, a.S - t1 * BM), lane);
    }
    for (int j = 0; j <= t0; ++j) {
      const int st = j % NST;
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_FULL + st), (j / NST) & 1, ctl, W_FWD_KV));
      if (ok) {
        const int nk = min(BN, a.S - j * BN);
        rows_to_atom(smem + OFF_KSC + st * 512, smem + OFF_KATOM + st * 512, nk, lane);
        cols_to_atom(smem + OFF_VSC + st * 512, smem + OFF_VATOM + st * 512, nk / 32, lane);
      }
      fence_proxy_async_smem();
      __syncwarp();
      named_sync(NB_KV, 64);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // ======================= softmax + epilogue: slot x, one query row per thread
    const int x = (warp - 4) >> 2;
    const int q = warp & 3;          // TMEM lane quarter
    const int r = q * 32 + lane;     // row inside the tile
    if (x == 0 || has1) {
      const int t = x == 0 ? t0 : t1, hq = x == 0 ? u.hq0 : u.hq1;
      const uint32_t lane_off = (uint32_t)(q * 32) << 16;
      const uint32_t tSx = tmem + T_S0 + 128u * x + lane_off, tOx = tmem + T_O0 + 128u * x + lane_off;
      const float sl2 = a.scale_log2e;
      uint32_t* patom = reinterpret_cast<uint32_t*>(smem + OFF_PATOM + x * 512 + lane * 16 + q * 4);
      // m: running row maximum of the scaled scores (log2 units), raised lazily; l: the row's sum of
      // 2^(s - m) over the keys so far.
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j <= t; ++j) {
        // does the MMA warp place the other slot's next QK scales in this S once it is loaded?
        const bool sl_needed = x == 1 ? (j < t0 && !(OWN && j == t1))
                                      : (j >= 1 && has1 && j <= t1 && !(OWN && j == t0));
        const bool diag = j == t;
        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_S_FULL + x), j & 1, ctl, W_SM_S));
        float v[128];
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) tld32(tSx + 32 * c, v + 32 * c);
          tmem_ld_wait();
        }
        if (sl_needed) {
          if (ok) {
            tc_fence_before();
            named_arrive(NB_SL + x, 32 + kSlotThreads);
          } else {
            named_sync(NB_SL + x, 32 + kSlotThreads);
          }
        }
        if (ok) {
          if (diag) {   // keys after the row (key index = column inside the diagonal tile)
#pragma unroll
            for (int k = 0; k < 128; ++k) v[k] = k > r ? -INFINITY : v[k];
          }
          // maxima of the four 32-key blocks and of the row
          float bm[4];
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const float* w = v + 32 * bb;
            float c0 = fmax3(w[0], w[1], w[2]), c1 = fmax3(w[3], w[4], w[5]);
            float c2 = fmax3(w[6], w[7], w[8]), c3 = fmax3(w[9], w[10], w[11]);
            c0 = fmax3(c0, w[12], w[13]);
            c1 = fmax3(c1, w[14], w[15]);
            c2 = fmax3(c2, w[16], w[17]);
            c3 = fmax3(c3, w[18], w[19]);
            c0 = fmax3(c0, w[20], w[21]);
            c1 = fmax3(c1, w[22], w[23]);
            c2 = fmax3(c2, w[24], w[25]);
            c3 = fmax3(c3, w[26], w[27]);
            c0 = fmax3(c0, w[28], w[29]);
            c1 = fmax3(c1, w[30], w[31]);
            bm[bb] = fmax3(c0, c1, fmaxf(c2, c3));
          }
          const float mt = fmax3(bm[0], bm[1], fmaxf(bm[2], bm[3])) * sl2;
          const bool need = mt > m + RESCALE_LOG2;   // true at j = 0
          if (j > 0 && __any_sync(0xFFFFFFFFu, need)) {
            // rescale this warp's O rows (factor 1 for rows that keep their maximum).  O is idle:
            // the S_FULL completion above implies that this slot's previous P.V has completed.
            const float alpha = need ? ex2_approx(m - mt) : 1.0f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t o[16];
              tmem_ld16(tOx + 16 * c, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tst16(tOx + 16 * c, o);
            }
            l *= alpha;
          }
          if (need) m = mt;
          // P relative to a power of two per 32-key block: 2^(x - m - e_b) with
          // e_b = floor(block max - m) - 7, so the block's largest weight lies in [2^7, 2^8) and no
          // element saturates the E4M3 range; the A scale of the P.V MMA for that block is 2^e_b.
          // The choice reads this row's own scores in the block only.
          int eb[4];
          float ad[4];
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const float tb = fmaxf(fmaf(bm[bb], sl2, -m), -300.f);
            eb[bb] = max(__float2int_rd(tb) - 7, -127);
            ad[bb] = -(m + (float)eb[bb]);
          }
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const float2 mul2 = make_float2(sl2, sl2), add2 = make_float2(ad[bb], ad[bb]);
            float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
            float* w = v + 32 * bb;
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
              const float2 xa = __ffma2_rn(make_float2(w[k], w[k + 1]), mul2, add2);
              const float2 xb = __ffma2_rn(make_float2(w[k + 2], w[k + 3]), mul2, add2);
              w[k] = ex2_approx(xa.x);
              w[k + 1] = ex2_approx(xa.y);
              w[k + 2] = ex2_approx(xb.x);
              w[k + 3] = ex2_approx(xb.y);
              s0 = __fadd2_rn(s0, make_float2(w[k], w[k + 1]));
              s1 = __fadd2_rn(s1, make_float2(w[k + 2], w[k + 3]));
            }
            l = fmaf(exp2i(eb[bb]), (s0.x + s0.y) + (s1.x + s1.y), l);
          }
          *patom = (uint32_t)(127 + eb[0]) | ((uint32_t)(127 + eb[1]) << 8) | ((uint32_t)(127 + eb[2]) << 16) |
                   ((uint32_t)(127 + eb[3]) << 24);
          // Per key block bb: E4M3 P (term 0) and, with two terms, the residual at the same scale
          // (term 1), word c holding keys 32bb + 4c .. 32bb + 4c + 3.  In the diagonal tile the own
          // block (bb == q, keys <= row) leaves the E4M3 P (its words are 0) and becomes BF16 P in
          // true weights 2^(x - m); key blocks after it are 0 already, and block 3, never a
          // completed block there, is not stored (its columns hold the P.V scales).
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const float* p = v + 32 * bb;
            const bool own_blk = OWN && diag && bb == q;   // warp-uniform
            uint32_t w0[8], w1[8];
            if (!own_blk) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint16_t h01 = cvt_e4m3x2(p[4 * c], p[4 * c + 1]), h23 = cvt_e4m3x2(p[4 * c + 2], p[4 * c + 3]);
                w0[c] = (uint32_t)h01 | ((uint32_t)h23 << 16);
                if (P_TERMS > 1) {
                  const uint32_t r01 = hsub2(pack_f16x2(p[4 * c], p[4 * c + 1]), cvt_e4m3x2_to_f16x2(h01));
                  const uint32_t r23 = hsub2(pack_f16x2(p[4 * c + 2], p[4 * c + 3]), cvt_e4m3x2_to_f16x2(h23));
                  w1[c] = (uint32_t)cvt_e4m3x2_f16x2(r01) | ((uint32_t)cvt_e4m3x2_f16x2(r23) << 16);
                }
              }
            } else {
#pragma unroll
              for (int c = 0; c < 8; ++c) w0[c] = w1[c] = 0u;
            }
            if (!(OWN && diag) || bb < 3) {
              tst8(tSx + 8 * bb, w0);
              if (P_TERMS > 1) tst8(tSx + C_P1 + 8 * bb, w1);
            }
            if (OWN && diag) {
              uint32_t own[16];
              if (own_blk) {
                const float sc = exp2i(eb[bb]);
#pragma unroll
                for (int k = 0; k < 16; ++k) own[k] = pack_bf16x2(p[2 * k] * sc, p[2 * k + 1] * sc);
              } else {
#pragma unroll
                for (int k = 0; k < 16; ++k) own[k] = 0u;
              }
              tst16(tSx + C_OWNP + 16 * bb, own);
            }
          }
        }
        if (ok) {
          fence_proxy_async_smem();   // the P scale atom, read by tcgen05.cp
          tmem_st_wait();
          tc_fence_before();
          named_arrive(NB_P + x, 32 + kSlotThreads);
        } else {
          named_sync(NB_P + x, 32 + kSlotThreads);
        }
      }
      // ---- epilogue: O / l -> BF16 (and/or MXFP8), LSE
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_O_FULL + x), 0, ctl, W_SM_O));
      if (ok) {
        tc_fence_after();
        const int i = t * BM + r;            // query token
        const bool row_ok = i < a.S;         // rows past S hold no token
        const float inv_l = 1.0f / l;
        const long long row = a.layout == 0 ? ((long long)b * a.S + i) * a.Hq + hq
                                            : ((long long)i * a.B + b) * a.Hq + hq;
        uint32_t scw = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tld32(tOx + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= inv_l;
          if (a.o != nullptr && row_ok) {
            uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) + row * HD + 32 * c);
#pragma unroll
            for (int e8 = 0; e8 < 4; ++e8) {
              orow[e8] = make_uint4(pack_bf16x2(o[8 * e8], o[8 * e8 + 1]), pack_bf16x2(o[8 * e8 + 2], o[8 * e8 + 3]),
                                    pack_bf16x2(o[8 * e8 + 4], o[8 * e8 + 5]),
                                    pack_bf16x2(o[8 * e8 + 6], o[8 * e8 + 7]));
            }
          }
          if (a.o8 != nullptr) {
            // MXFP8 O: the 32 columns of chunk c are the row's 32-element block c, so the block
            // maximum is thread-local.  The maximum is taken on |bit patterns| (NaN above Inf above
            // every finite value).
            uint32_t mb = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) mb = max(mb, __float_as_uint(o[e]) & 0x7FFFFFFFu);
            float inv;
            const uint32_t sbyte = e8m0_from_amax(__uint_as_float(mb), inv);
            uint32_t wq[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t lo = cvt_e4m3x2(o[4 * k] * inv, o[4 * k + 1] * inv);
              const uint32_t hi = cvt_e4m3x2(o[4 * k + 2] * inv, o[4 * k + 3] * inv);
              wq[k] = sbyte == 0xFFu ? 0x7F7F7F7Fu : (lo | (hi << 16));
            }
            if (row_ok) {
              uint4* dst = reinterpret_cast<uint4*>(a.o8 + row * HD + 32 * c);
              dst[0] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
              dst[1] = make_uint4(wq[4], wq[5], wq[6], wq[7]);
            }
            scw |= sbyte << (8 * c);
          }
        }
        if (row_ok) {
          const long long srow = ((long long)b * a.Hq + hq) * a.S + i;
          if (a.o8 != nullptr) *reinterpret_cast<uint32_t*>(a.o_sc + srow * 4) = scw;
          a.lse[srow] = (m + lg2_approx(l)) * 0.69314718055994531f;
        }
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
  auto kern = attn_fwd_kernel<P_TERMS, LEAKY>;
  // the attribute is per function and per device; set it once per device
  static unsigned long long set_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&set_mask, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&set_mask, bit, __ATOMIC_ACQ_REL);
  }
  const long long T = (args.S + BM - 1) / BM;
  const long long pairs = (T * (args.Hq / args.Hkv) + 1) / 2;
  const long long ctas = (long long)args.B * args.Hkv * pairs;
  kern<<<(unsigned)ctas, kThreads, SMEM_BYTES, st>>>(args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnArgs& args, cudaStream_t st) {
  if (args.p_terms == 2) return args.leaky ? launch_variant<2, true>(args, st) : launch_variant<2, false>(args, st);
  return args.leaky ? launch_variant<1, true>(args, st) : launch_variant<1, false>(args, st);
}

}  // namespace bsc
