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
// Warp roles (256 threads):
//   warp 0      TMA producer: the Q tile with its compact scales once; K and V (columnwise,
//               transposed) tiles with their compact scales through a 4-stage ring.
//   warp 1      allocates TMEM; its elected lane issues tcgen05.cp (scale factors, Q) and tcgen05.mma.
//   warp 2      decodes the own-block tile of the token-normalised V to BF16 (exact).
//   warp 3      waits for each K/V stage and permutes its compact scales into the tensor cores'
//               scale-factor atoms.
//   warps 4-7   softmax, one query row per thread (TMEM 32x32b shape), then the epilogue.
// The scores are double-buffered in TMEM and P (E4M3, 32 columns per term) is written over the S
// buffer it came from.  The QK MMA of tile j + 2 follows the P.V of tile j into the same buffer, so
// the scores of the next tile are ready when the softmax of a tile ends: the softmax runs tile
// after tile without waiting for an MMA, and the tensor cores work behind it.
// TMEM (512 columns): S[0] 0-127, S[1] 128-255, O 256-383, Q 384-415 (E4M3, the QK MMA's A
// operand), scale factors 480-507.  In the diagonal tile the own-block BF16 P takes 64 columns of
// the other S buffer once the previous tile's P.V has read it.
// The MMA-issuing thread waits on hardware named barriers only: an mbarrier wait in that thread
// returns only once its MMAs in flight have completed, a named barrier does not.  Every mbarrier
// wait elsewhere is bounded, and every role passes every named-barrier generation, also after an
// abort, so no named barrier can wait forever.
#include <cstdint>
#include <type_traits>
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
constexpr int NST = 4;    // K/V shared-memory stages (the producer's wait rule assumes 4)
// Softmax sets: with one E4M3 term for P, one set of four softmax warps takes every key tile; with two
// terms (more exponent and convert work per tile) two sets of four take alternate tiles (set x the
// tiles j with j mod 2 == x, so always S[x]), handing the running row maximum to each other.
template <int P_TERMS> constexpr int kSets = P_TERMS == 2 ? 2 : 1;
template <int P_TERMS> constexpr int kThreadsFor = 128 + 128 * kSets<P_TERMS>;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t TILE8 = BM * HD;                      // one 128 x 128 E4M3 tile
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE8;                // NST stages, 128 keys x 128 d
constexpr uint32_t OFF_V = OFF_K + NST * TILE8;          // NST stages, 128 d rows x 128 keys
constexpr uint32_t OFF_VT = OFF_V + NST * TILE8;         // own-block V, BF16 [key][d], two 64-d blocks
constexpr uint32_t OFF_QSC = OFF_VT + 2 * BN * HD;       // compact Q scales
constexpr uint32_t OFF_QATOM = OFF_QSC + 512;            // Q scale atom
constexpr uint32_t OFF_KSC = OFF_QATOM + 512;            // compact K scales, NST stages
constexpr uint32_t OFF_VSC = OFF_KSC + NST * 512;        // compact V scales, NST stages
constexpr uint32_t OFF_KATOM = OFF_VSC + NST * 512;      // K scale atoms, NST stages
constexpr uint32_t OFF_VATOM = OFF_KATOM + NST * 512;    // V scale atoms, NST stages
constexpr uint32_t OFF_BAR = OFF_VATOM + NST * 512;
constexpr uint32_t NUM_BARS = 32;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;    // tmem slot, abort flag
constexpr uint32_t OFF_MROW = OFF_MISC + 16;             // per row: the running maximum last decided
constexpr uint32_t OFF_LROW = OFF_MROW + 512;            // per row: set 1's part of the row sum
constexpr uint32_t SMEM_USED = OFF_LROW + 512;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;        // alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// mbarriers (phase k of a per-tile barrier belongs to key tile k):
//   Q_FULL        the Q tile and its scales landed
//   FULL[st]      stage st's K, V tiles and compact scales landed (producer's copies)
//   S_FULL[b]     the scores of tile j are in S[b] (and every earlier MMA has completed: the
//                 P.V of tiles j - 2 and before, so also the last reader of tile j - 2's K/V
//                 stage; and for j >= 1 the P.V of tile j - 1 once tile j + 1's scores are in)
//   P_DONE        the P.V of the tile before the diagonal tile has completed (its S buffer may
//                 take the own-block P; O is idle)
//   O_FULL        O is final; VT_READY: the own-block V tile is decoded
enum Bar : uint32_t {
  B_Q_FULL = 0,
  B_FULL = 1,                    // + stage
  B_S_FULL = B_FULL + NST,       // + buffer
  B_P_DONE = B_S_FULL + 2,
  B_O_FULL,
  B_VT_READY,
  B_DRAIN,
  B_INJECT,
  B_COUNT,
};
static_assert(B_COUNT <= NUM_BARS, "barrier slots");

// TMEM columns
constexpr uint32_t T_S0 = 0, T_S1 = 128, T_O = 256, T_Q = 384, T_SFQ = 480, T_SFK = 484, T_SFV = 492,
                   T_SFP = 500;   // SFK, SFV, SFP: two sets of 4 columns (tile parity)
constexpr uint32_t C_P1 = 32;    // the second P term's columns inside the S buffer
static_assert(T_SFP + 8 <= 512, "TMEM columns");

// The running row maximum m (log2 units) is raised only when a tile's maximum exceeds it by more
// than RESCALE_LOG2; O and l are then rescaled.  P carries a power-of-two scale per row and 32-key
// block, so the lag costs no E4M3 range.
constexpr float RESCALE_LOG2 = 8.0f;

// wait-site codes reported through the device status word
enum Site : int {
  W_PROD_FREE = 1, W_MMA_Q, W_FWD_KV, W_MMA_VT, W_MMA_INJECT,
  W_SM_S, W_SM_PV, W_SM_O, W_DEC_VTN, W_FWD_Q, W_MMA_KV, W_MMA_P, W_TMEM_BASE,
};

// Named barriers (ID 0 is __syncthreads):
//   NB_KV      forwarder + MMA warp, once per key tile, both blocking: the stage's tiles landed and
//              its scale atoms are written (the first generation covers the Q tile as well);
//   NB_P + (j mod 3)   softmax warps (arrive) + MMA warp (sync): the P of tile j and its scales are
//              written.  Three IDs in turn: the scores of tile j + 2, and so its arrivals, exist
//              only after the MMA warp has passed tile j's generation; and a softmax warp that
//              gives up at tile j (a failed wait; it then blocks on every later generation) has
//              arrived without waiting up to tile j - 1 at most, whose scores imply that the MMA
//              warp has passed tile j - 3.  So no sync or arrival can ever join the generation of
//              another tile.  With two IDs a warp giving up mid-run could join tile j - 2's
//              generation while a slower warp had not yet arrived there, and a random-interleaving
//              model of that protocol then deadlocked.
constexpr uint32_t NB_KV = 1, NB_P = 2, kPIds = 3;
constexpr uint32_t kNbP = 32 + 32 * 4;   // the MMA warp and the four softmax warps of the tile's set
//   NB_M + (j mod 2)   (two sets) the set that owns tile j (arrive) + the other set (sync): the row
//              maximum decided at tile j is in shared memory.  Each set takes the previous tile's
//              decision before it publishes its own, so the decisions of consecutive tiles alternate
//              between the two IDs and a generation never holds arrivals of two tiles.
//   NB_L       (two sets) set 1 (arrive) + set 0 (sync): set 1's part of the row sum is in shared memory.
constexpr uint32_t NB_M = 5, NB_L = 7, kNbM = 256;
static_assert(NB_L < 16, "named barrier IDs");

__device__ __forceinline__ float pow2_e8m0(uint32_t sb) {
  return sb == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(sb << 23);   // 2^(sb-127), sb <= 254
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

// P of one row of a key tile, per 32-key block: 2^(x - m - e_b) with e_b = floor(block max - m) - 7,
// so the block's largest weight lies in [2^7, 2^8) (exactly 2^7 for the block holding the running
// maximum) and no element saturates E4M3; the A scale of the P.V MMA for the block is 2^e_b (byte
// 127 + e_b, returned packed, byte b for block b).  Only this row's own scores in the block enter,
// so no scale depends on another row or on a key the row cannot see.  Word c of block b holds keys
// 32b + 4c .. 32b + 4c + 3; with two terms, w1 holds the E4M3 residual at the same scale.
// OWN_DIAG (the diagonal tile of the leak-free method): the own block b == q (keys <= row) leaves
// the E4M3 P (its words are 0) and becomes BF16 P in weights 2^(x - m) in `own`; key blocks after
// it are 0 already.  Adds the row's weights to l.
template <int P_TERMS, bool OWN_DIAG>
__device__ __forceinline__ uint32_t block_p(float (&v)[128], const float (&bm)[4], float m, float sl2, int q,
                                            uint32_t (&w0)[32], uint32_t (&w1)[32], uint32_t (&own)[16], float& l) {
  uint32_t sfw = 0;
#pragma unroll
  for (int bb = 0; bb < 4; ++bb) {
    const int e = max(__float2int_rd(fmaxf(fmaf(bm[bb], sl2, -m), -300.f)) - 7, -127);
    sfw |= (uint32_t)(127 + e) << (8 * bb);
    const float bscale = exp2i(e);
    const float2 mul2 = make_float2(sl2, sl2), add2 = make_float2(-(m + (float)e), -(m + (float)e));
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
    float* w = v + 32 * bb;
    if (OWN_DIAG && bb == q) {   // warp-uniform
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float2 xa = __ffma2_rn(make_float2(w[4 * c], w[4 * c + 1]), mul2, add2);
        const float2 xb = __ffma2_rn(make_float2(w[4 * c + 2], w[4 * c + 3]), mul2, add2);
        const float2 pa = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
        const float2 pb = make_float2(ex2_approx(xb.x), ex2_approx(xb.y));
        s0 = __fadd2_rn(s0, pa);
        s1 = __fadd2_rn(s1, pb);
        own[2 * c] = pack_bf16x2(pa.x * bscale, pa.y * bscale);
        own[2 * c + 1] = pack_bf16x2(pb.x * bscale, pb.y * bscale);
        w0[8 * bb + c] = 0u;
        w1[8 * bb + c] = 0u;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float2 xa = __ffma2_rn(make_float2(w[4 * c], w[4 * c + 1]), mul2, add2);
        const float2 xb = __ffma2_rn(make_float2(w[4 * c + 2], w[4 * c + 3]), mul2, add2);
        const float2 pa = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
        const float2 pb = make_float2(ex2_approx(xb.x), ex2_approx(xb.y));
        s0 = __fadd2_rn(s0, pa);
        s1 = __fadd2_rn(s1, pb);
        const uint16_t h01 = cvt_e4m3x2(pa.x, pa.y), h23 = cvt_e4m3x2(pb.x, pb.y);
        w0[8 * bb + c] = (uint32_t)h01 | ((uint32_t)h23 << 16);
        if (P_TERMS > 1) {
          const uint32_t r01 = hsub2(pack_f16x2(pa.x, pa.y), cvt_e4m3x2_to_f16x2(h01));
          const uint32_t r23 = hsub2(pack_f16x2(pb.x, pb.y), cvt_e4m3x2_to_f16x2(h23));
          w1[8 * bb + c] = (uint32_t)cvt_e4m3x2_f16x2(r01) | ((uint32_t)cvt_e4m3x2_f16x2(r23) << 16);
        }
      }
    }
    l = fmaf(bscale, (s0.x + s0.y) + (s1.x + s1.y), l);
  }
  return sfw;
}

template <int P_TERMS, bool LEAKY>
__global__ void __launch_bounds__(kThreadsFor<P_TERMS>, 1) attn_fwd_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int SETS = kSets<P_TERMS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](uint32_t i) { return sbase + OFF_BAR + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  constexpr bool OWN = !LEAKY;   // the own block goes through the token-normalised V

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (a.S + BM - 1) / BM;   // the last tile may hold fewer rows (S is a multiple of 32)
  // heaviest tiles first; the query heads sharing a KV head are adjacent
  const int bh = (int)(blockIdx.x % (unsigned)(a.B * a.Hq));
  const int t = T - 1 - (int)(blockIdx.x / (unsigned)(a.B * a.Hq));
  const int hq = bh % a.Hq, b = bh / a.Hq;
  const int hk = hq / (a.Hq / a.Hkv);
  const long long kv_plane = (long long)b * a.Hkv + hk;

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(B_FULL + s), 1);
    }
    mbar_init(bar(B_S_FULL + 0), 1);
    mbar_init(bar(B_S_FULL + 1), 1);
    mbar_init(bar(B_P_DONE), 1);
    mbar_init(bar(B_O_FULL), 1);
    mbar_init(bar(B_VT_READY), 1);
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
  const WaitCtl ctl{abort_flag, a.dev_status, a.limit_ns};
  // The CTA holds all 512 columns of the SM's tensor memory, so the allocation starts at lane 0,
  // column 0 and every TMEM address below is a compile-time constant (operands of tcgen05.mma then
  // need no per-instruction register moves).  Checked: a different base aborts the call.
  constexpr uint32_t tmem = 0;
  if (threadIdx.x == 0 && *tmem_slot != 0u) {
    *abort_flag = 1;
    if (a.dev_status) atomicCAS(a.dev_status, 0, 0x100 | W_TMEM_BASE);
  }
  __syncthreads();
  const bool start_ok = *abort_flag == 0;

  // Two sets: the launch gives 168 registers per thread (384 x 168 = 64512); the four helper warps keep
  // 112, the eight softmax warps get 192: 128 x 112 + 256 x 192 = 63488.
  if (warp < 4) {
  if constexpr (SETS == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
  if (warp == 0) {
    // ======================= producer
    if (lane == 0) {
      prefetch_tensormap(&a.tm_q);
      prefetch_tensormap(&a.tm_k);
      prefetch_tensormap(&a.tm_v);
      const int nr = min(BM, a.S - t * BM);
      mbar_arrive_expect_tx(bar(B_Q_FULL), TILE8 + 4u * (uint32_t)nr);
      tma_load_4d(sbase + OFF_Q, &a.tm_q, bar(B_Q_FULL), 0, hq, t * BM, b);
      bulk_load(sbase + OFF_QSC, a.q_sc + (((long long)b * a.Hq + hq) * a.S + (long long)t * BM) * 4, 4u * (uint32_t)nr,
                bar(B_Q_FULL));
      int nl[NST] = {};   // stage loads issued
      bool ok = start_ok;
      for (int j = 0; j <= t && ok; ++j) {
        const int st = j % NST;
        // Before loading tile j (j >= 2) wait for the scores of tile j - 2.  From j = 4 on this is
        // what frees stage st: its last reader, the P.V of tile j - 4, was issued before them.
        // At j = 2, 3 it keeps this thread's parity waits unambiguous: each buffer's phases are
        // then observed in order, and phase k + 2 cannot complete before tile j is loaded.
        if (j >= 2 && !(ok = mbar_wait(bar(B_S_FULL + (j & 1)), ((j - 2) >> 1) & 1, ctl, W_PROD_FREE))) break;
        const uint32_t nk = (uint32_t)min(BN, a.S - j * BN);
        // K and V tiles; K scales (nk words) and V scales (nk / 32 blocks of 128 bytes) compact
        mbar_arrive_expect_tx(bar(B_FULL + st), 2 * TILE8 + 8u * nk);
        tma_load_4d(sbase + OFF_K + st * TILE8, &a.tm_k, bar(B_FULL + st), 0, hk, j * BN, b);
        bulk_load(sbase + OFF_KSC + st * 512, a.k_sc + (kv_plane * a.S + (long long)j * BN) * 4, 4u * nk,
                  bar(B_FULL + st));
        tma_load_2d(sbase + OFF_V + st * TILE8, &a.tm_v, bar(B_FULL + st), j * BN, (int)(kv_plane * HD));
        bulk_load(sbase + OFF_VSC + st * 512, a.v_sc + (kv_plane * (a.S / 32) + (long long)j * 4) * 128, 4u * nk,
                  bar(B_FULL + st));
        ++nl[st];
      }
      // drain: every copy this thread issued must land before the CTA may exit
      for (int st = 0; st < NST; ++st) {
        if (nl[st] > 0) mbar_wait_drain(bar(B_FULL + st), (nl[st] - 1) & 1, a.limit_ns);
      }
      mbar_wait_drain(bar(B_Q_FULL), 0, a.limit_ns);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer: lane 0 issues, the whole warp meets the named barriers.
    // Every generation is met, also after an abort (then nothing is issued).
    const uint64_t dK = desc_kmajor_sw128(sbase + OFF_K), dV = desc_kmajor_sw128(sbase + OFF_V);
    const uint32_t tO = tmem + T_O;
    bool ok = start_ok;
    if (lane == 0 && a.inject_stall) ok = mbar_wait(bar(B_INJECT), 0, ctl, W_MMA_INJECT);   // nothing arrives here
    // S[j % 2] = Q K_j^T (Q from TMEM)
    auto qk = [&](int j) {
      const int st = j % NST, sb = j & 1;
      tc_cp_32x128b_warpx4(tmem + T_SFK + 4 * sb, desc_sf_block(sbase + OFF_KATOM + st * 512));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_mxf8_ts(tmem + (sb ? T_S1 : T_S0), tmem + T_Q + 8 * kk, dK + (uint64_t)(st * (TILE8 / 16) + 2 * kk),
                    idesc_mxf8(BM, BN, kk, kk), tmem + T_SFQ, tmem + T_SFK + 4 * sb, kk > 0 ? 1u : 0u);
      }
      tc_commit(bar(B_S_FULL + sb));
    };
    // O += P_j V_j (completed blocks, E4M3, P over S[j % 2]); OWN_TILE (the diagonal tile of the
    // leak-free method): key block 3 is never a completed block there and is not read at all, and
    // the own block follows (BF16, P in the other S buffer).  No runtime branch sits between the
    // MMAs of one group.
    auto pv = [&](int j, auto own_tile) {
      constexpr bool OWN_TILE = decltype(own_tile)::value;
      const int st = j % NST, sb = j & 1;
      const uint32_t tPs = tmem + (sb ? T_S1 : T_S0), sfa = tmem + T_SFP + 4 * sb, sfb = tmem + T_SFV + 4 * sb;
      const uint64_t dVs = dV + (uint64_t)(st * (TILE8 / 16));
      const uint32_t acc0 = j > 0 ? 1u : 0u;
      tc_cp_32x128b_warpx4(sfb, desc_sf_block(sbase + OFF_VATOM + st * 512));
#pragma unroll
      for (int term = 0; term < P_TERMS; ++term) {
#pragma unroll
        for (int kk = 0; kk < (OWN_TILE ? 3 : 4); ++kk) {
          mma_mxf8_ts(tO, tPs + term * C_P1 + 8 * kk, dVs + 2 * kk, idesc_mxf8(BM, HD, kk, kk), sfa, sfb,
                      (term > 0 || kk > 0) ? 1u : acc0);
        }
      }
      if (OWN_TILE) {
        ok = mbar_wait(bar(B_VT_READY), 0, ctl, W_MMA_VT);   // once per CTA
        if (ok) {
          tc_fence_after();
          const uint32_t tPo = tmem + (((t + 1) & 1) ? T_S1 : T_S0);   // own-block BF16 P
#pragma unroll
          for (int s = 0; s < 8; ++s) {   // B is [key][d]: MN-major, 16 keys = 2048 bytes per step
            mma_f16_ts(tO, tPo + 8 * s, smem_desc(sbase + OFF_VT + s * 2048, 16384, 1024, 2),
                       idesc_bf16(BM, HD) | (1u << 16), 1u);
          }
        }
      }
      if (j == t - 1) tc_commit(bar(B_P_DONE));   // the own-block P goes over this tile's S next
    };
    named_sync(NB_KV, 64);   // Q and K/V tile 0
    if (lane == 0 && ok) {
      tc_fence_after();
      tc_cp_32x128b_warpx4(tmem + T_SFQ, desc_sf_block(sbase + OFF_QATOM));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {   // Q into TMEM, 32 bytes of each row per copy
        asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(tmem + T_Q + 8 * kk),
                     "l"(desc_kmajor_sw128(sbase + OFF_Q) + 2 * kk)
                     : "memory");
      }
      qk(0);
    }
    __syncwarp();   // the warp meets each barrier converged
    if (t >= 1) {
      named_sync(NB_KV, 64);
      if (lane == 0 && ok) {
        tc_fence_after();
        qk(1);
      }
      __syncwarp();
    }
    uint32_t pid = NB_P;   // NB_P + j mod kPIds
    for (int j = 0; j <= t; ++j) {
      named_sync(pid, kNbP);
      pid = pid == NB_P + kPIds - 1 ? NB_P : pid + 1;
      if (lane == 0 && ok) {
        tc_fence_after();
        if (j < t) {
          pv(j, std::false_type{});
        } else {
          if (OWN) pv(j, std::true_type{});
          else pv(j, std::false_type{});
          tc_commit(bar(B_O_FULL));
        }
      }
      __syncwarp();
      if (j + 2 <= t) {
        // S[j % 2] is rewritten after P.V of tile j has read it (the MMAs run in issue order)
        named_sync(NB_KV, 64);
        if (lane == 0 && ok) {
          tc_fence_after();
          qk(j + 2);
        }
        __syncwarp();
      }
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
    if (OWN) {
      const int nkeys = min(BN, a.S - t * BN);
      uint8_t* dst = smem + OFF_VT;
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
      if (lane == 0) mbar_arrive(bar(B_VT_READY));
    }
  } else if (warp == 3) {
    // ======================= forwarder: compact scales -> scale-factor atoms, stage by stage, then a
    // named-barrier generation with the MMA warp (every generation is met, also after an abort)
    bool ok = start_ok && __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_Q_FULL), 0, ctl, W_FWD_Q));
    if (ok) rows_to_atom(smem + OFF_QSC, smem + OFF_QATOM, min(BM, a.S - t * BM), lane);
    for (int j = 0; j <= t; ++j) {
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
    if constexpr (SETS == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // ======================= softmax + epilogue: one query row per thread; set x takes the key tiles
    // j with j mod SETS == x; set 0 writes the output
    const int x = SETS == 2 ? (warp - 4) >> 2 : 0;
    const int q = warp & 3;          // TMEM lane quarter
    const int r = q * 32 + lane;     // row inside the tile
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sl2 = a.scale_log2e;
    // m: running row maximum of the scaled scores (log2 units), raised lazily, as last decided (by
    // either set); l: this set's part of the row's sum of 2^(s - m) over its keys so far.
    float m = -INFINITY, l = 0.f;
    bool ok = start_ok;
    uint32_t pid = NB_P + x;   // NB_P + j mod kPIds for this set's tile j
    float* m_row = reinterpret_cast<float*>(smem + OFF_MROW);
    float* l_row = reinterpret_cast<float*>(smem + OFF_LROW);
    // (two sets) take the maximum decided at tile jj by the other set; this set's sum follows a raise
    auto msync = [&](int jj) {
      named_sync(NB_M + (jj & 1), kNbM);
      const float mp = m_row[r];
      if (mp > m) {
        l *= ex2_approx(m - mp);
        m = mp;
      }
    };
    // One key tile.  The diagonal tile (DIAG) has its own instantiation, peeled out of the loop, so
    // that the loop body holds only the code of ordinary tiles.
    auto tile = [&](int j, auto diag_tag) {
      constexpr bool DIAG = decltype(diag_tag)::value;
      const int sb = j & 1;
      // one pass of work; a failed wait leaves it early (break), the tile's barrier generations are
      // still met below, in the same order
      bool published = false;
      do {
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_S_FULL + sb), (j >> 1) & 1, ctl, W_SM_S));
      if (!ok) break;
      tc_fence_after();
      float v[128];
      float bm[4];   // maxima of the four 32-key blocks
      if constexpr (!DIAG) {
        // every key of the tile is visible to every row: each load returns its block's maximum too
#pragma unroll
        for (int c = 0; c < 4; ++c) tld32_max(tmem + lane_off + (sb ? T_S1 : T_S0) + 32 * c, v + 32 * c, bm[c]);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) tld32(tmem + lane_off + (sb ? T_S1 : T_S0) + 32 * c, v + 32 * c);
        tmem_ld_wait();
        // keys after the row (key index = column inside the diagonal tile), then the block maxima
#pragma unroll
        for (int k = 0; k < 128; ++k) v[k] = k > r ? -INFINITY : v[k];
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
      }
      if (SETS == 2 && j > 0) msync(j - 1);
      const float mt = fmax3(bm[0], bm[1], fmaxf(bm[2], bm[3])) * sl2;
      const bool need = mt > m + RESCALE_LOG2;   // true at j = 0
      const float m_new = need ? mt : m;
      if constexpr (SETS == 2) {   // publish this tile's decision for the other set's next tile
        m_row[r] = m_new;
        __threadfence_block();
        named_arrive(NB_M + (j & 1), kNbM);
        published = true;
      }
      if (j > 0 && __any_sync(0xFFFFFFFFu, need)) {
        // rescale this warp's O rows (factor 1 for rows that keep m) once the previous P.V, the
        // last writer of O, has completed: the scores of tile j + 1 are computed after it (the
        // diagonal tile has none; P_DONE marks it there)
        if (!(ok = __all_sync(0xFFFFFFFFu, j < t ? mbar_wait(bar(B_S_FULL + ((j + 1) & 1)), ((j + 1) >> 1) & 1, ctl, W_SM_PV)
                                                  : mbar_wait(bar(B_P_DONE), 0, ctl, W_SM_PV))))
          break;
        tc_fence_after();
        const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[16];
          tmem_ld16(tmem + lane_off + T_O + 16 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tst16(tmem + lane_off + T_O + 16 * c, o);
        }
        l *= alpha;
      }
      m = m_new;
      uint32_t w0[32], w1[32], own[16];
      uint32_t sfw;
      if constexpr (OWN && DIAG) sfw = block_p<P_TERMS, true>(v, bm, m, sl2, q, w0, w1, own, l);
      else sfw = block_p<P_TERMS, false>(v, bm, m, sl2, q, w0, w1, own, l);
      // P over this tile's S buffer (its scores are in registers); the S_FULL completion above
      // implies that the P.V two tiles back, the last reader of the buffer and of this parity's
      // scale columns, has completed
      const uint32_t tP = tmem + lane_off + (sb ? T_S1 : T_S0);
      if constexpr (OWN && DIAG) {
        tst16(tP, w0);
        tst8(tP + 16, w0 + 16);
        if (P_TERMS > 1) {
          tst16(tP + C_P1, w1);
          tst8(tP + C_P1 + 16, w1 + 16);
        }
        // own-block BF16 P into the other S buffer, once the previous tile's P.V has read it
        if (t > 0 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_P_DONE), 0, ctl, W_SM_PV)))) break;
        tc_fence_after();
        const uint32_t tPo = tmem + lane_off + (((t + 1) & 1) ? T_S1 : T_S0);
        const uint32_t zero16[16] = {};
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          if (bb == q) tst16(tPo + 16 * bb, own);
          else tst16(tPo + 16 * bb, zero16);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) tst8(tP + 8 * c, w0 + 8 * c);
        if (P_TERMS > 1) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tst8(tP + C_P1 + 8 * c, w1 + 8 * c);
        }
      }
      // row r's four block scales: lane r, column T_SFP + 4 sb + r / 32 (the cell the MMA reads)
      asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tmem + lane_off + T_SFP + 4 * sb + q),
                   "r"(sfw)
                   : "memory");
      tmem_st_wait();
      } while (false);
      // P of this tile is written (or this warp gave up: then, with two sets, it still takes the
      // previous tile's maximum and publishes one, in that order, and it blocks on the P generation,
      // so that it can never arrive on a later generation before the MMA warp has passed this one)
      if (SETS == 2 && !published) {
        if (j > 0) msync(j - 1);
        named_arrive(NB_M + (j & 1), kNbM);
      }
      if (ok) {
        tc_fence_before();
        named_arrive(pid, kNbP);
      } else {
        named_sync(pid, kNbP);
      }
      if constexpr (SETS == 2) pid = pid >= NB_P + 1 ? pid - 1 : pid + 2;   // tile j + 2
      else pid = pid == NB_P + kPIds - 1 ? NB_P : pid + 1;
    };
    for (int j = x; j < t; j += SETS) tile(j, std::false_type{});
    if (SETS == 1 || (t & 1) == x) tile(t, std::true_type{});
    else msync(t);   // the final maximum, decided by the other set
    if constexpr (SETS == 2) {   // set 1's part of the row sum (relative to the final maximum) to set 0
      if (x == 1) {
        l_row[r] = l;
        __threadfence_block();
        named_arrive(NB_L, kNbM);
      } else {
        named_sync(NB_L, kNbM);
        l += l_row[r];
      }
    }
    // ---- epilogue (set 0): O / l -> BF16 (and/or MXFP8), LSE
    if (x != 0) ok = false;
    if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(B_O_FULL), 0, ctl, W_SM_O));
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
        tld32(tmem + lane_off + T_O + 32 * c, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] *= inv_l;
        if (a.o != nullptr && row_ok) {
          uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) + row * HD + 32 * c);
#pragma unroll
          for (int e8 = 0; e8 < 4; ++e8) {
            orow[e8] = make_uint4(pack_bf16x2(o[8 * e8], o[8 * e8 + 1]), pack_bf16x2(o[8 * e8 + 2], o[8 * e8 + 3]),
                                  pack_bf16x2(o[8 * e8 + 4], o[8 * e8 + 5]), pack_bf16x2(o[8 * e8 + 6], o[8 * e8 + 7]));
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

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(*tmem_slot, 512);
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
  const long long ctas = (long long)args.B * args.Hq * ((args.S + BM - 1) / BM);
  kern<<<(unsigned)ctas, kThreadsFor<P_TERMS>, SMEM_BYTES, st>>>(args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnArgs& args, cudaStream_t st) {
  if (args.p_terms == 2) return args.leaky ? launch_variant<2, true>(args, st) : launch_variant<2, false>(args, st);
  return args.leaky ? launch_variant<1, true>(args, st) : launch_variant<1, false>(args, st);
}

}  // namespace bsc
