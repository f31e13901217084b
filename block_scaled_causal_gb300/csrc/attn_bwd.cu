// Backward of the leak-free causal MXFP8 attention, on decoded operands, with BF16 tensor-core MMAs.
//
// "[PyTorch] Add causal MXFP8 attention without future-token leakage through V scales"
// (TransformerEngine PR #3865), Description, Backward: an FP16/BF16 attention backward on Q and K
// decoded from their rowwise MXFP8 bytes and V decoded from the token-normalised copy, fed with
// the forward's O and LSE, so no gradient depends on a future token.  With s = scale * Qh Kh^T:
//   P = exp(s - LSE),  dV = P^T dO,  dP = dO Vt^T,  Dlt = rowsum(dO * O),  dS = P * (dP - Dlt),
//   dQ = scale * dS Kh,  dK = scale * dS^T Qh;  a KV head's dK, dV sum over its query heads.
//
// Two launches:
//   * prep: decodes Qh, Kh and Vt to BF16 planes [B][H][Sp][D] in the caller's workspace (rows
//     past S zero) and writes the row statistics Dlt and LSE log2(e) there, once per call;
//   * one grid of two CTA roles:
//     - dK/dV: one CTA per (batch, KV head, 128-key tile); walks the group's (query head, query
//       tile) pairs at or after the key tile, accumulating dV and dK in tensor memory;
//     - dQ: one CTA per (batch, query head, 128-row query tile); walks the key tiles up to the
//       diagonal, accumulating dQ in tensor memory.
// Both roles are warp-specialised (384 threads): warp 0 lane 0 issues the copies, warp 1 lane 0 the
// MMAs, warps 4-11 compute P and dS (two warps per TMEM lane quarter, each with half the columns of
// its rows); warps 2-3 take part in the epilogue only.  Every MMA is BF16.  P and dS reach their MMAs
// from tensor memory (written there by the softmax warps); dQ keeps Qh and dO in tensor memory as
// A operands, dK/dV keeps Kh and Vt in shared memory (so that its S^T and dP^T get N = 128).  Every tile
// sits in shared memory in its natural orientation ([row][column], 64-column blocks with the
// 128-byte swizzle); the products that contract over its rows (P^T dO, dS^T Qh, dS Kh) read it as
// an MN-major operand, so nothing is transposed.  Every mbarrier wait is bounded; the MMA-issuing
// thread waits on named barriers only (an mbarrier wait there drains its MMAs in flight).
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bsc_internal.h"
#include "ptx.cuh"

namespace bsc {
namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // keys per tile
constexpr int HD = 128;   // head dimension
constexpr uint32_t ATOM = 128 * 128;   // one 128-row x 128-byte swizzle block (64 BF16 columns)
constexpr uint32_t TILE = 2 * ATOM;    // a 128 x 128 BF16 tile
static_assert(BM == 128 && BN == 128 && HD == 128, "tile shapes assumed by the tensor-memory layouts");

enum Site : int {
  W_TMEM_BASE = 0x20, W_MMA_LD, W_PROD, W_SM_LD, W_SM_S, W_SM_DP, W_EPI,
};

// A wait's outcome made the same for every thread of the CTA.
__device__ __forceinline__ bool cta_all(bool ok) { return __syncthreads_and(ok ? 1 : 0) != 0; }

// ------------------------------------------------------------------------------------------------
// E4M3 -> BF16 without the conversion unit.  A byte's sign placed at bit 15 and its seven other
// bits (exponent and mantissa) at bits 4-10 of a BF16 give the byte's value times 2^-120 for every
// code, subnormals included: the BF16 exponent field then holds the E4M3 one, whose bias is 120
// less, and BF16 subnormals continue the E4M3 subnormal spacing.  Two exact BF16 multiplications
// (2^120, then the block's power-of-two scale) finish the decode.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
  return r;
}
// t holds two bytes at bits 0-7 and 16-23 (other bits zero) -> BF16x2 of their values x 2^-120.
__device__ __forceinline__ uint32_t e4m3x2_times_2m120(uint32_t t) {
  const uint32_t u = t << 4;                  // magnitude bits at 4-10, sign at bit 11
  const uint32_t sgn = u & 0x08000800u;
  return u + sgn * 15u;                       // the sign moves from bit 11 to bit 15
}
// BF16x2 of the E8M0 scale 2^(sb - 127) (sb = 0: 2^-127, a BF16 subnormal).
__device__ __forceinline__ uint32_t bf16x2_pow2_e8m0(uint32_t sb) {
  const uint32_t h = sb == 0 ? 0x0040u : (sb << 7);
  return h | (h << 16);
}
// Four E4M3 bytes (element e in byte e) times scale2 (BF16x2) -> four BF16 (one uint2).
__device__ __forceinline__ uint2 decode4_bf16(uint32_t x, uint32_t scale2) {
  constexpr uint32_t kTwo120 = 0x7B807B80u;   // 2^120 in both halves
  return make_uint2(bf16x2_mul(bf16x2_mul(e4m3x2_times_2m120(__byte_perm(x, 0u, 0x4140)), kTwo120), scale2),
                    bf16x2_mul(bf16x2_mul(e4m3x2_times_2m120(__byte_perm(x, 0u, 0x4342)), kTwo120), scale2));
}

// ------------------------------------------------------------------------------------------------
// prep.  Grid (Sp / 64, B * Hq, 4): block z picks the job, y the (batch, head) plane, x a run of
// 64 rows; each of the 8 warps takes 8 rows, with every load of its rows issued before any is used.
//   z = 0, 1, 2: Qh, Kh, Vt rows: 128 E4M3 bytes -> 128 BF16; 8 lanes per row, lane l taking bytes
//     16 l..16 l + 15, whose scale is the row's block l / 2 (Q and K rowwise scales) or V's one
//     amplitude per token; a warp takes 4 rows per pass.  Planes past B * Hkv are idle for Kh and Vt;
//   z = 3: statistics: Dlt_i = <dO_i, O_i> (fp32; lane l sums elements 4l..4l+3, then a butterfly
//     over the warp) and LSE_i log2(e).
// Rows at or past S: zero BF16 rows, Dlt = 0 and LSE = +inf, which make their P and dS exactly 0.
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const __grid_constant__ BwdArgs a) {
  const int lane = threadIdx.x & 31, job = blockIdx.z;
  const int plane = blockIdx.y;   // b * H + h
  const int H = job == 0 || job == 3 ? a.Hq : a.Hkv;
  if (plane >= a.B * H) return;
  const int b = plane / H, h = plane - b * H;
  const int i0 = blockIdx.x * 64 + (threadIdx.x >> 5) * 8;
  const long long prow = (long long)plane * a.Sp;   // the plane's first row in the workspace
  auto src_row = [&](int i) {
    return a.layout == 0 ? ((long long)b * a.S + i) * H + h : ((long long)i * a.B + b) * H + h;
  };
  if (job < 3) {
    const uint8_t* src = job == 0 ? a.q8 : job == 1 ? a.k8 : a.vtn;
    uint16_t* dst = job == 0 ? a.qh : job == 1 ? a.kh : a.vh;
    const int r4 = lane >> 3, l8 = lane & 7;
    uint4 x[2];
    uint32_t sb[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = i0 + 4 * k + r4;
      x[k] = make_uint4(0u, 0u, 0u, 0u);
      sb[k] = 0u;
      if (i < a.S) {
        x[k] = __ldg(reinterpret_cast<const uint4*>(src + src_row(i) * HD) + l8);
        sb[k] = job == 2 ? __ldg(a.vtn_sc + (long long)plane * a.S + i)
                         : __ldg((job == 0 ? a.q_sc : a.k_sc) + ((long long)plane * a.S + i) * 4 + (l8 >> 1));
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = i0 + 4 * k + r4;
      uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
      if (i < a.S) {
        const uint32_t s2 = bf16x2_pow2_e8m0(sb[k]);
        const uint2 d0 = decode4_bf16(x[k].x, s2), d1 = decode4_bf16(x[k].y, s2);
        const uint2 d2 = decode4_bf16(x[k].z, s2), d3 = decode4_bf16(x[k].w, s2);
        lo = make_uint4(d0.x, d0.y, d1.x, d1.y);
        hi = make_uint4(d2.x, d2.y, d3.x, d3.y);
      }
      uint4* out = reinterpret_cast<uint4*>(dst + (prow + i) * HD) + 2 * l8;
      out[0] = lo;
      out[1] = hi;
    }
    return;
  }
  const long long plane_rows = (long long)a.B * a.Hq * a.Sp;
  uint2 xo[8], yo[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = i0 + k;
    xo[k] = yo[k] = make_uint2(0u, 0u);
    if (i < a.S) {
      const long long row = src_row(i);
      xo[k] = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.o) + row * HD) + lane);
      yo[k] = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.dO) + row * HD) + lane);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = i0 + k;
    float acc = 0.f;
    const uint32_t xs[2] = {xo[k].x, xo[k].y}, ys[2] = {yo[k].x, yo[k].y};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      acc = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), acc);
      acc = fmaf(__uint_as_float(xs[e] & 0xFFFF0000u), __uint_as_float(ys[e] & 0xFFFF0000u), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) {
      a.ws[prow + i] = i < a.S ? acc : 0.f;
      a.ws[plane_rows + prow + i] = i < a.S ? a.lse[(long long)plane * a.S + i] * 1.4426950408889634f : INFINITY;
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Shared pieces of the two attention kernels.

// Epilogue: an accumulator (128 rows x 128 columns fp32 in TMEM) times `mul` -> BF16 rows of a
// tensor laid out like Q (BSHD/SBHD with H heads); rows at or past S are not written.  8 warps:
// warp w reads lanes 32 (w % 4).. and columns 64 (w / 4)..
__device__ __forceinline__ void store_acc(uint32_t tmem_acc, void* out, const BwdArgs& a, int H, int b, int h,
                                          int tile, float mul) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qq = warp & 3, half = warp >> 2;
  const int r = qq * 32 + lane;
  const int i = tile * BM + r;
  float o[64];
  const uint32_t ta = tmem_acc + ((uint32_t)(qq * 32) << 16) + 64 * half;
  tld32(ta, o);
  tld32(ta + 32, o + 32);
  tmem_ld_wait();
  if (i >= a.S) return;
  const long long row = a.layout == 0 ? ((long long)b * a.S + i) * H + h : ((long long)i * a.B + b) * H + h;
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + row * HD + 64 * half);
#pragma unroll
  for (int e8 = 0; e8 < 8; ++e8) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(o[8 * e8 + 2 * e] * mul, o[8 * e8 + 2 * e + 1] * mul);
    dst[e8] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// A 128 x 128 BF16 tile of a workspace plane (rows `row0`.., plane `plane`) into shared memory:
// two 64-column boxes, the 128-byte swizzle.
__device__ __forceinline__ void load_plane_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar, int row0,
                                                long long plane) {
  tma_load_3d(dst, map, bar, 0, row0, (int)plane);
  tma_load_3d(dst + ATOM, map, bar, 64, row0, (int)plane);
}
// The same for dO (the caller's tensor, 4-D map {D, Hq, S, B}).
__device__ __forceinline__ void load_do_tile(uint32_t dst, const BwdArgs& a, uint32_t bar, int hq, int row0, int b) {
  tma_load_4d(dst, &a.tm_do, bar, 0, hq, row0, b);
  tma_load_4d(dst + ATOM, &a.tm_do, bar, 64, hq, row0, b);
}
// A BF16 tile in shared memory (K-major, 128-byte swizzle) into 64 TMEM columns: the A-operand
// layout, K = 16 elements (8 columns) per MMA step.
__device__ __forceinline__ void tile_to_tmem(uint32_t tcol, uint32_t src) {
#pragma unroll
  for (int s = 0; s < 8; ++s) tc_cp_128x256b(tcol + 8 * s, desc_kmajor_sw128(src + (s >> 2) * ATOM + (s & 3) * 32));
}
// D (+)= A B^T over K = 16 * NSTEP, A in TMEM (8 columns per step from t_a), B in shared memory:
// K-major (the next 32 bytes of a row, 64-column blocks ATOM apart) or MN-major (the next 16
// rows, 2048 bytes; LBO = ATOM between the 64-column blocks of N).
template <int NSTEP, bool B_MN>
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t t_a, uint64_t b_desc, uint32_t idesc, uint32_t acc0) {
#pragma unroll
  for (int s = 0; s < NSTEP; ++s) {
    const uint32_t off = B_MN ? (uint32_t)s * (2048 >> 4) : (uint32_t)(((s >> 2) * ATOM + (s & 3) * 32) >> 4);
    mma_f16_ts(d, t_a + 8 * s, b_desc + off, idesc, s > 0 ? 1u : acc0);
  }
}
// dS = P (dP - Dlt) of 32 columns, packed to BF16 pairs (Dlt in 16-byte shared-memory loads, the
// same address in every lane).
__device__ __forceinline__ void ds_chunk(const float* p, const float* d, const float* dlt, uint32_t* w) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 dl = *reinterpret_cast<const float4*>(dlt + 4 * i);
    w[2 * i] = pack_bf16x2(p[4 * i] * (d[4 * i] - dl.x), p[4 * i + 1] * (d[4 * i + 1] - dl.y));
    w[2 * i + 1] = pack_bf16x2(p[4 * i + 2] * (d[4 * i + 2] - dl.z), p[4 * i + 3] * (d[4 * i + 3] - dl.w));
  }
}

// ================================================================================================
// dK, dV.  One CTA per (batch, KV head hk, 128-key tile jt); it walks the pairs n = 0..N-1 of (query
// head of the group, query tile at or after jt): query tiles from the last down, the group's heads
// innermost, so CTAs of one KV head running together read the same Qh and dO tiles from L2.  The
// keys sit on the TMEM lanes, so P^T and dS^T are the A operands of the dV and dK MMAs straight from
// tensor memory:
//   S^T  = Kh Qh^T      (M = 128 keys, N = 128 queries; A = Kh and B = Qh from shared memory)
//   dP^T = Vt dO^T      (A = Vt, B = dO from shared memory)
//   P^T  = exp2(S^T scale log2(e) - LSE2[q]),  dS^T = P^T (dP^T - Dlt[q])     (softmax warps)
//   dV  += P^T dO       A = P^T (BF16 in S^T's columns), B = dO read along q
//   dK  += dS^T Qh      A = dS^T (BF16 in dP^T's columns), B = Qh read along q
// Kh and Vt stay in shared memory, so S^T and dP^T get 128 columns each (an MMA of N = 128 does
// twice the work of one of N = 64 in about 1.25x the time).  Eight softmax warps: those of one TMEM
// lane quarter take 64 queries each (warps 4-7 queries 0-63, warps 8-11 queries 64-127) and write
// their BF16 P^T and dS^T over their own columns (queries 64 h.. at columns 64 h..64 h+31): the A
// operands in two K halves.  MMA issue order S(0) dP(0) | dV(n) S(n+1) dK(n) dP(n+1) | ...: the
// softmax of pair n + 1 runs under dK(n) and dP(n + 1), its dS under dV(n + 1) and S(n + 2).  An MMA
// that rewrites columns an earlier one reads (S(n+1) over P^T(n), dP(n+1) over dS^T(n)) is issued
// after it: the MMAs of one thread run in issue order.  TMEM: S^T 0-127, dP^T 128-255, dV 256-383,
// dK 384-511.
constexpr uint32_t KV_KH = 0;            // Kh bf16 [key][d]
constexpr uint32_t KV_VH = TILE;         // Vt bf16 [key][d]
constexpr uint32_t KV_QH = 2 * TILE;     // 2 stages: Qh bf16 [q][d]
constexpr uint32_t KV_DO = 4 * TILE;     // 2 stages: dO bf16 [q][d]
constexpr uint32_t KV_STAT = 6 * TILE;   // 2 stages: Dlt[128], then LSE2[128]
constexpr uint32_t KV_BAR = KV_STAT + 2048;
constexpr uint32_t KV_MISC = KV_BAR + 128;   // TMEM slot, abort flag
constexpr uint32_t KV_SMEM = KV_MISC + 16 + 1024;
static_assert(KV_SMEM <= 227 * 1024, "shared memory budget");
constexpr uint32_t T_ST = 0, T_DPT = 128, T_DV = 256, T_DK = 384;
constexpr int kThreadsKv = 384;
// mbarriers:
//   KV        Kh and Vt landed
//   LF + st   Qh, dO and the statistics of a pair landed in stage st
//   SF        S^T(n) computed (and every MMA issued before it)
//   DP        dP^T(n) computed
//   PD + st   the MMAs of the pair in stage st have completed (up to its dK)
enum KvBar : uint32_t { KB_KV = 0, KB_LF = 1, KB_SF = 3, KB_DP, KB_PD, KB_DRAIN = KB_PD + 2, KB_COUNT };
static_assert(KB_COUNT * 8 <= 128, "barrier slots");
// Named barriers, softmax warps (256 threads) + MMA warp (32):
//   NB_LD   a pair's data landed (the softmax warps wait for the copies; once per pair)
//   NB_P    P^T(n) is in TMEM
//   NB_DS   dS^T(n) is in TMEM
// The softmax warps block on NB_DS and arrive on the others: each blocking generation they pass
// shows the MMA warp has passed the previous generation of every barrier they arrive on next, so no
// generation ever holds arrivals of two pairs, also once a role has given up (a failed wait: it
// skips its work but meets every generation).  Both sides meet the generations in one order.
constexpr uint32_t NB_LD = 1, NB_P = 2, NB_DS = 3, kNb = 256 + 32;

// One dK/dV CTA; `cta` is its index among them.  `a` is the kernel's grid-constant parameter (the
// tensor maps are read from there).
__device__ __forceinline__ void dkdv_cta(const BwdArgs& a, int cta) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](uint32_t i) { return sbase + KV_BAR + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + KV_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + KV_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int T = (a.S + BN - 1) / BN;
  const int g = a.Hq / a.Hkv;
  // key tiles with the most query tiles first
  const int bh = cta % (a.B * a.Hkv);
  const int jt = cta / (a.B * a.Hkv);
  const int hk = bh % a.Hkv, b = bh / a.Hkv;
  const long long kv_plane = (long long)b * a.Hkv + hk;
  const int N = g * (T - jt);   // pairs; the last g of them are the diagonal tile
  auto hq_of = [&](int n) { return hk * g + n % g; };
  auto it_of = [&](int n) { return T - 1 - n / g; };

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < KB_COUNT; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + KV_MISC, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The CTA holds all 512 columns, so the allocation starts at column 0 and every TMEM address is
  // a compile-time constant.  Checked: a different base aborts the call.
  constexpr uint32_t tmem = 0;
  if (threadIdx.x == 0 && *tmem_slot != 0u) {
    *abort_flag = 1;
    if (a.dev_status) atomicCAS(a.dev_status, 0, 0x100 | W_TMEM_BASE);
  }
  __syncthreads();
  const bool start_ok = *abort_flag == 0;
  const WaitCtl ctl{abort_flag, a.dev_status, a.limit_ns};

  if (warp == 0) {
    // ======================= copies
    if (lane == 0) {
      prefetch_tensormap(&a.tm_qh);
      prefetch_tensormap(&a.tm_kh);
      prefetch_tensormap(&a.tm_vh);
      prefetch_tensormap(&a.tm_do);
      const long long ws_plane = (long long)a.B * a.Hq * a.Sp;
      auto load_pair = [&](int n) {
        const int st = n & 1, it = it_of(n), hq = hq_of(n);
        const long long qplane = (long long)b * a.Hq + hq, srow = qplane * a.Sp + (long long)it * BM;
        const uint32_t fb = bar(KB_LF + st);
        mbar_arrive_expect_tx(fb, 2 * TILE + 1024);
        load_plane_tile(sbase + KV_QH + st * TILE, &a.tm_qh, fb, it * BM, qplane);
        load_do_tile(sbase + KV_DO + st * TILE, a, fb, hq, it * BM, b);
        bulk_load(sbase + KV_STAT + st * 1024, a.ws + srow, 512, fb);
        bulk_load(sbase + KV_STAT + st * 1024 + 512, a.ws + ws_plane + srow, 512, fb);
      };
      bool ok = start_ok;
      int nl[2] = {0, 0};
      if (ok) {
        mbar_arrive_expect_tx(bar(KB_KV), 2 * TILE);
        load_plane_tile(sbase + KV_KH, &a.tm_kh, bar(KB_KV), jt * BN, kv_plane);
        load_plane_tile(sbase + KV_VH, &a.tm_vh, bar(KB_KV), jt * BN, kv_plane);
        for (int n = 0; n < 2 && n < N; ++n) {
          load_pair(n);
          nl[n] = 1;
        }
      }
      // stage n % 2 takes pair n + 2 once the MMAs of pair n have completed: they were its last
      // readers, and the softmax warps were done with its statistics before its dK
      for (int n = 0; ok && n + 2 < N; ++n) {
        if (!(ok = mbar_wait(bar(KB_PD + (n & 1)), (uint32_t)(n >> 1) & 1u, ctl, W_PROD))) break;
        load_pair(n + 2);
        ++nl[n & 1];
      }
      // every copy this thread issued lands before the CTA may exit
      if (start_ok) mbar_wait_drain(bar(KB_KV), 0, a.limit_ns);
      for (int st = 0; st < 2; ++st)
        if (nl[st] > 0) mbar_wait_drain(bar(KB_LF + st), (uint32_t)(nl[st] - 1) & 1u, a.limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer: lane 0 issues, the whole warp meets the named barriers
    bool ok = start_ok;
    if (lane == 0 && ok) ok = mbar_wait(bar(KB_KV), 0, ctl, W_MMA_LD);   // nothing in flight yet
    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
    auto live = [&]() { return ok && *abort_flag == 0; };
    const uint64_t dKk = desc_kmajor_sw128(sbase + KV_KH), dVk = desc_kmajor_sw128(sbase + KV_VH);
    const uint64_t dQk = desc_kmajor_sw128(sbase + KV_QH), dDOk = desc_kmajor_sw128(sbase + KV_DO);
    const uint64_t dQm = smem_desc(sbase + KV_QH, ATOM, 1024, 2), dDOm = smem_desc(sbase + KV_DO, ATOM, 1024, 2);
    constexpr uint32_t idN = idesc_bf16(BN, BM), idMN = idesc_bf16(BN, HD) | (1u << 16);
    auto stg = [](int n) { return (uint32_t)(((n & 1) * TILE) >> 4); };
    // D = A B^T over d, both K-major in shared memory
    auto mma_ss = [&](uint32_t d, uint64_t da, uint64_t db) {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t off = (uint32_t)(((s >> 2) * ATOM + (s & 3) * 32) >> 4);
        mma_f16_ss(d, da + off, db + off, idN, s > 0 ? 1u : 0u);
      }
    };
    // D (+)= A B over the pair's 128 queries: A in TMEM at columns 0-31 (queries 0-63) and 64-95
    // (queries 64-127), B read along q
    auto mma_q = [&](uint32_t d, uint32_t t_a, uint64_t db, uint32_t acc0) {
      mma_ts<4, true>(d, t_a, db, idMN, acc0);
      mma_ts<4, true>(d, t_a + 64, db + 4 * (2048 >> 4), idMN, 1u);
    };
    auto issue_s = [&](int n) {
      mma_ss(tmem + T_ST, dKk, dQk + stg(n));
      tc_commit(bar(KB_SF));
    };
    auto issue_dp = [&](int n) {
      mma_ss(tmem + T_DPT, dVk, dDOk + stg(n));
      tc_commit(bar(KB_DP));
    };
    named_sync(NB_LD, kNb);
    if (lane == 0 && live()) {
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    __syncwarp();
    for (int n = 0; n < N; ++n) {
      named_sync(NB_P, kNb);
      if (lane == 0 && live()) {   // dV += P^T dO
        tc_fence_after();
        mma_q(tmem + T_DV, tmem + T_ST, dDOm + stg(n), n > 0 ? 1u : 0u);
      }
      __syncwarp();
      if (n + 1 < N) {
        named_sync(NB_LD, kNb);   // the next pair's data
        if (lane == 0 && live()) {
          tc_fence_after();
          issue_s(n + 1);
        }
        __syncwarp();
      }
      named_sync(NB_DS, kNb);
      if (lane == 0 && live()) {   // dK += dS^T Qh
        tc_fence_after();
        mma_q(tmem + T_DK, tmem + T_DPT, dQm + stg(n), n > 0 ? 1u : 0u);
        tc_commit(bar(KB_PD + (n & 1)));
        if (n + 1 < N) issue_dp(n + 1);
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(bar(KB_DRAIN));   // every MMA of the CTA
    __syncwarp();
  } else if (warp >= 4) {
    // ======================= softmax: key row kr of the tile per thread, queries 64 h.. of it
    const int qq = warp & 3, kr = qq * 32 + lane, h = (warp - 4) >> 2;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const uint32_t col = 64 * h;   // this warp's columns of S^T and dP^T
    const float sl2 = a.scale_log2e;
    bool ok = start_ok;
    // pair n's data landed; then its generation of NB_LD.  The first is met blocking: the arrival
    // for pair 1 then follows the MMA warp's passing of pair 0's generation also when a wait failed.
    auto landed = [&](int n) {
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_LF + (n & 1)), (uint32_t)(n >> 1) & 1u, ctl, W_SM_LD));
      if (n == 0) named_sync(NB_LD, kNb);
      else named_arrive(NB_LD, kNb);
    };
    auto pair = [&](int n, auto diag_tag) {
      constexpr bool DIAG = decltype(diag_tag)::value;
      const float* dlt = reinterpret_cast<const float*>(smem + KV_STAT + (n & 1) * 1024) + 64 * h;
      const float* lse2 = dlt + 128;
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_SF), (uint32_t)n & 1u, ctl, W_SM_S));
      float p[64];
      if (ok) {
        tc_fence_after();
        tld32(tmem + lane_off + T_ST + col, p);
        tld32(tmem + lane_off + T_ST + col + 32, p + 32);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 l = *reinterpret_cast<const float4*>(lse2 + 4 * q4);
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = 4 * q4 + e;
            const float x = ex2_approx(fmaf(p[q], sl2, -lv[e]));
            p[q] = (DIAG && 64 * h + q < kr) ? 0.f : x;   // in the diagonal tile a query sees keys up to itself
          }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(p[32 * c + 2 * i], p[32 * c + 2 * i + 1]);
          tst16(tmem + lane_off + T_ST + col + 16 * c, w);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      named_arrive(NB_P, kNb);
      if (n + 1 < N) landed(n + 1);
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_DP), (uint32_t)n & 1u, ctl, W_SM_DP));
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {   // dS^T of queries 64 h + 32 c.. over columns 64 h + 16 c.., read by then
          float d[32];
          uint32_t w[16];
          tld32(tmem + lane_off + T_DPT + col + 32 * c, d);
          tmem_ld_wait();
          ds_chunk(p + 32 * c, d, dlt + 32 * c, w);
          tst16(tmem + lane_off + T_DPT + col + 16 * c, w);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      named_sync(NB_DS, kNb);
    };
    landed(0);
    int n = 0;
    for (; n < N - g; ++n) pair(n, std::false_type{});
    for (; n < N; ++n) pair(n, std::true_type{});
  }

  // ======================= epilogue: dV and dK from TMEM, 8 warps
  tc_fence_before();
  __syncthreads();
  const bool drained = mbar_wait_drain(bar(KB_DRAIN), 0, a.limit_ns);
  tc_fence_after();
  if (cta_all(drained && start_ok && *abort_flag == 0) && warp < 8) {
    store_acc(tmem + T_DV, a.dv, a, a.Hkv, b, hk, jt, 1.0f);
    store_acc(tmem + T_DK, a.dk, a, a.Hkv, b, hk, jt, a.scale);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ================================================================================================
// dQ.  One CTA per (batch, query head hq, 128-row query tile it); key tiles j = 0..it, the diagonal
// tile last.  Qh and dO of the tile stay in tensor memory as the A operands:
//   S   = Qh Kh_j^T     (B = Kh [key][d], K-major)
//   dP  = dO Vt_j^T     (B = Vt [key][d], K-major)
//   P   = exp2(S scale log2(e) - LSE2),  dS = P (dP - Dlt)     (softmax warps, one query row each)
//   dQ += dS Kh_j       A = dS (BF16 over dP's columns 0-31 and 64-95), B = Kh read along the keys
// Issue order S(0) dP(0) | S(j+1) dQ(j) dP(j+1) | ...: S(j+1) follows as soon as the softmax warps
// have read S(j) (P stays in registers), so P(j+1) runs under dQ(j) and dP(j+1), and dS(j+1) under
// S(j+2).  dP(j+1) rewrites the columns dQ(j) reads and is issued after it.
// TMEM: Qh 0-63, dO 64-127, S 128-255, dP 256-383, dQ 384-511.
// Key tiles go round three shared-memory stages of 64 KB (Kh, then Vt); Qh and dO arrive in stage
// 2, which takes its first key tile (tile 2) once they have been copied into TMEM.
constexpr int KST = 3;                      // key-tile stages
constexpr uint32_t QQ_STAGE = 2 * TILE;     // stage s at s * QQ_STAGE: Kh bf16 [key][d], then Vt
constexpr uint32_t QQ_QH = 2 * QQ_STAGE;    // Qh bf16 [q][d], then dO: in stage 2 at the start
constexpr uint32_t QQ_DO = QQ_QH + TILE;
constexpr uint32_t QQ_STAT = KST * QQ_STAGE;   // Dlt[128], then LSE2[128]
constexpr uint32_t QQ_BAR = QQ_STAT + 1024;
constexpr uint32_t QQ_MISC = QQ_BAR + 128;   // TMEM slot, abort flag
constexpr uint32_t QQ_SMEM = QQ_MISC + 16 + 1024;
static_assert(QQ_SMEM <= 227 * 1024, "shared memory budget");
constexpr uint32_t T_QH = 0, T_DOH = 64, T_S = 128, T_DP = 256, T_DQ = 384;
// mbarriers: QD (Qh, dO and the statistics of the tile), CP (Qh and dO copied into TMEM), KF + s (a
// key tile's Kh and Vt landed in stage s), SF (S(j) computed), DP (dP(j) computed), KD + s (the
// MMAs of the key tile in stage s have completed, up to dQ(j)).
enum QBar : uint32_t {
  QB_QD = 0, QB_CP, QB_KF, QB_SF = QB_KF + KST, QB_DP, QB_KD, QB_DRAIN = QB_KD + KST, QB_COUNT
};
static_assert(QB_COUNT * 8 <= 128, "barrier slots");
// Named barriers, softmax warps (256) + MMA warp (32), with the rules of the dK/dV kernel:
//   NB_LD  a key tile landed;  NB_S  S(j) has been read;  NB_DS  dS(j) is in TMEM (blocking).
// 12 warps: the softmax work of a query row is split between two warps of the same TMEM lane
// quarter (warps 4-7 keys 0-63, warps 8-11 keys 64-127); each writes its dS over its own dP
// columns (keys 64 kh.. at columns 64 kh..64 kh+31), the A operand of dQ in two K halves.
constexpr int kThreadsDq = 384;
constexpr uint32_t kNbDq = 256 + 32;
constexpr uint32_t NB_S = 2;

// One dQ CTA; `cta` is its index among them.
__device__ __forceinline__ void dq_cta(const BwdArgs& a, int cta) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](uint32_t i) { return sbase + QQ_BAR + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + QQ_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + QQ_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int T = (a.S + BM - 1) / BM;
  const int bh = cta % (a.B * a.Hq);
  const int it = T - 1 - cta / (a.B * a.Hq);   // heaviest query tiles first
  const int hq = bh % a.Hq, b = bh / a.Hq;
  const int hk = hq / (a.Hq / a.Hkv);
  const long long kv_plane = (long long)b * a.Hkv + hk, q_plane = (long long)b * a.Hq + hq;
  const int J = it + 1;   // key tiles

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < QB_COUNT; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + QQ_MISC, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  constexpr uint32_t tmem = 0;   // all 512 columns, checked as in the dK/dV kernel
  if (threadIdx.x == 0 && *tmem_slot != 0u) {
    *abort_flag = 1;
    if (a.dev_status) atomicCAS(a.dev_status, 0, 0x100 | W_TMEM_BASE);
  }
  __syncthreads();
  const bool start_ok = *abort_flag == 0;
  const WaitCtl ctl{abort_flag, a.dev_status, a.limit_ns};

  if (warp == 0) {
    // ======================= copies
    if (lane == 0) {
      prefetch_tensormap(&a.tm_qh);
      prefetch_tensormap(&a.tm_kh);
      prefetch_tensormap(&a.tm_vh);
      prefetch_tensormap(&a.tm_do);
      auto load_kv = [&](int j) {
        const int st = j % KST;
        const uint32_t fb = bar(QB_KF + st);
        mbar_arrive_expect_tx(fb, 2 * TILE);
        load_plane_tile(sbase + st * QQ_STAGE, &a.tm_kh, fb, j * BN, kv_plane);
        load_plane_tile(sbase + st * QQ_STAGE + TILE, &a.tm_vh, fb, j * BN, kv_plane);
      };
      bool ok = start_ok;
      int nl[KST] = {0, 0, 0};
      if (ok) {
        const long long srow = q_plane * a.Sp + (long long)it * BM;
        mbar_arrive_expect_tx(bar(QB_QD), 2 * TILE + 1024);
        load_plane_tile(sbase + QQ_QH, &a.tm_qh, bar(QB_QD), it * BM, q_plane);
        load_do_tile(sbase + QQ_DO, a, bar(QB_QD), hq, it * BM, b);
        bulk_load(sbase + QQ_STAT, a.ws + srow, 512, bar(QB_QD));
        bulk_load(sbase + QQ_STAT + 512, a.ws + (long long)a.B * a.Hq * a.Sp + srow, 512, bar(QB_QD));
        for (int j = 0; j < 2 && j < J; ++j) {
          load_kv(j);
          nl[j] = 1;
        }
        // stage 2 once Qh and dO have been copied out of it
        if (J > 2 && (ok = mbar_wait(bar(QB_CP), 0, ctl, W_PROD))) {
          load_kv(2);
          nl[2] = 1;
        }
      }
      // stage j % 3 takes key tile j + 3 once the MMAs of tile j (its last readers) have completed
      for (int j = 0; ok && j + KST < J; ++j) {
        if (!(ok = mbar_wait(bar(QB_KD + j % KST), (uint32_t)(j / KST) & 1u, ctl, W_PROD))) break;
        load_kv(j + KST);
        ++nl[j % KST];
      }
      if (start_ok) mbar_wait_drain(bar(QB_QD), 0, a.limit_ns);
      for (int st = 0; st < KST; ++st)
        if (nl[st] > 0) mbar_wait_drain(bar(QB_KF + st), (uint32_t)(nl[st] - 1) & 1u, a.limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer
    bool ok = start_ok;
    if (lane == 0 && ok) {   // Qh and dO into TMEM (nothing is in flight yet)
      ok = mbar_wait(bar(QB_QD), 0, ctl, W_MMA_LD);
      if (ok) {
        tc_fence_after();
        tile_to_tmem(tmem + T_QH, sbase + QQ_QH);
        tile_to_tmem(tmem + T_DOH, sbase + QQ_DO);
        tc_commit(bar(QB_CP));
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
    auto live = [&]() { return ok && *abort_flag == 0; };
    const uint64_t dKk = desc_kmajor_sw128(sbase), dVk = desc_kmajor_sw128(sbase + TILE);
    const uint64_t dKm = smem_desc(sbase, ATOM, 1024, 2);
    constexpr uint32_t idN = idesc_bf16(BM, BN), idMN = idesc_bf16(BM, HD) | (1u << 16);
    auto soff = [](int j) { return (uint32_t)(((j % KST) * QQ_STAGE) >> 4); };
    auto issue_s = [&](int j) {
      mma_ts<8, false>(tmem + T_S, tmem + T_QH, dKk + soff(j), idN, 0u);
      tc_commit(bar(QB_SF));
    };
    auto issue_dp = [&](int j) {
      mma_ts<8, false>(tmem + T_DP, tmem + T_DOH, dVk + soff(j), idN, 0u);
      tc_commit(bar(QB_DP));
    };
    named_sync(NB_LD, kNbDq);
    if (lane == 0 && live()) {
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    __syncwarp();
    for (int j = 0; j < J; ++j) {
      named_sync(NB_S, kNbDq);
      if (j + 1 < J) {
        named_sync(NB_LD, kNbDq);
        if (lane == 0 && live()) {
          tc_fence_after();
          issue_s(j + 1);
        }
        __syncwarp();
      }
      named_sync(NB_DS, kNbDq);
      if (lane == 0 && live()) {   // dQ += dS Kh
        tc_fence_after();
        mma_ts<4, true>(tmem + T_DQ, tmem + T_DP, dKm + soff(j), idMN, j > 0 ? 1u : 0u);
        mma_ts<4, true>(tmem + T_DQ, tmem + T_DP + 64, dKm + soff(j) + 4 * (2048 >> 4), idMN, 1u);
        tc_commit(bar(QB_KD + j % KST));
        if (j + 1 < J) issue_dp(j + 1);
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(bar(QB_DRAIN));
    __syncwarp();
  } else if (warp >= 4) {
    // ======================= softmax: query row r of the tile per thread, keys 64 kh.. of it
    const int qq = warp & 3, r = qq * 32 + lane, kh = (warp - 4) >> 2;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const float sl2 = a.scale_log2e;
    bool ok = start_ok;
    if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(QB_QD), 0, ctl, W_SM_LD));
    const float dlt = ok ? reinterpret_cast<const float*>(smem + QQ_STAT)[r] : 0.f;
    const float lse2 = ok ? reinterpret_cast<const float*>(smem + QQ_STAT)[128 + r] : 0.f;
    // key tile j landed; then its generation of NB_LD.  The first is met blocking: the arrival for
    // tile 1 then follows the MMA warp's passing of tile 0's generation also when a wait failed.
    auto landed = [&](int j) {
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(QB_KF + j % KST), (uint32_t)(j / KST) & 1u, ctl, W_SM_LD));
      if (j == 0) named_sync(NB_LD, kNbDq);
      else named_arrive(NB_LD, kNbDq);
    };
    auto tile = [&](int j, auto diag_tag) {
      constexpr bool DIAG = decltype(diag_tag)::value;
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(QB_SF), (uint32_t)j & 1u, ctl, W_SM_S));
      float p[64];
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) tld32(tmem + lane_off + T_S + 64 * kh + 32 * c, p + 32 * c);
        tmem_ld_wait();
        tc_fence_before();
      }
      named_arrive(NB_S, kNbDq);   // S(j) is in registers: S(j+1) may be computed over it
      if (j + 1 < J) landed(j + 1);   // and, once its tile landed, issued right away
      if (ok) {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const float x = ex2_approx(fmaf(p[k], sl2, -lse2));
          p[k] = (DIAG && 64 * kh + k > r) ? 0.f : x;   // in the diagonal tile a query sees keys up to itself
        }
      }
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(QB_DP), (uint32_t)j & 1u, ctl, W_SM_DP));
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {   // dS of keys 64 kh + 32c.. over columns 64 kh + 16c.., read by then
          float d[32];
          uint32_t w[16];
          tld32(tmem + lane_off + T_DP + 64 * kh + 32 * c, d);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(p[32 * c + 2 * i] * (d[2 * i] - dlt), p[32 * c + 2 * i + 1] * (d[2 * i + 1] - dlt));
          tst16(tmem + lane_off + T_DP + 64 * kh + 16 * c, w);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      named_sync(NB_DS, kNbDq);
    };
    landed(0);
    for (int j = 0; j < J - 1; ++j) tile(j, std::false_type{});
    tile(J - 1, std::true_type{});
  }

  // ======================= epilogue: dQ from TMEM, 8 warps
  tc_fence_before();
  __syncthreads();
  const bool drained = mbar_wait_drain(bar(QB_DRAIN), 0, a.limit_ns);
  tc_fence_after();
  if (cta_all(drained && start_ok && *abort_flag == 0) && warp < 8) store_acc(tmem + T_DQ, a.dq, a, a.Hq, b, hq, it, a.scale);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}


// dK/dV and dQ in one grid: the dK/dV CTAs (heaviest key tiles first), then the dQ CTAs (heaviest
// query tiles first).  The two are independent once the prep kernel has run; in one grid the CTAs
// of one fill the SMs the other's last CTAs leave idle.
static_assert(kThreadsKv == kThreadsDq, "one block size for both roles");
constexpr uint32_t BWD_SMEM = KV_SMEM > QQ_SMEM ? KV_SMEM : QQ_SMEM;
__global__ void __launch_bounds__(kThreadsKv, 1) attn_bwd_kernel(const __grid_constant__ BwdArgs a) {
  const int T = (a.S + BN - 1) / BN;
  const int nkv = a.B * a.Hkv * T;
  if ((int)blockIdx.x < nkv) dkdv_cta(a, (int)blockIdx.x);
  else dq_cta(a, (int)blockIdx.x - nkv);
}

}  // namespace

size_t bwd_workspace_bytes(int B, int S, int Hq, int Hkv) {
  const size_t Sp = (size_t)((S + BM - 1) / BM) * BM;
  return (size_t)B * Sp * (8 * (size_t)Hq + 2 * HD * ((size_t)Hq + 2 * (size_t)Hkv));
}

cudaError_t launch_attn_bwd(const BwdArgs& args, cudaStream_t st) {
  static bool attr_set = false;   // the attribute is per function and per process
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BWD_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long T = (args.S + BM - 1) / BM;
  if ((long long)args.B * args.Hq > 65535) return cudaErrorInvalidConfiguration;   // the prep grid's y
  attn_bwd_prep_kernel<<<dim3((unsigned)(args.Sp / 64), (unsigned)(args.B * args.Hq), 4), 256, 0, st>>>(args);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long ctas = (long long)args.B * (args.Hkv + args.Hq) * T;
  if (ctas >= (1LL << 31)) return cudaErrorInvalidConfiguration;
  attn_bwd_kernel<<<(unsigned)ctas, kThreadsKv, BWD_SMEM, st>>>(args);
  return cudaGetLastError();
}

}  // namespace bsc
