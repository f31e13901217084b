// Backward of the leak-free causal MXFP8 attention, on decoded operands, with BF16 tensor-core MMAs.
//
// "[PyTorch] Add causal MXFP8 attention without future-token leakage through V scales"
// (TransformerEngine PR #3865), Description, Backward: an FP16/BF16 attention backward on Q and K
// decoded from their rowwise MXFP8 bytes and V decoded from the token-normalised copy, fed with
// the forward's O and LSE, so no gradient depends on a future token.  With s = scale * Qh Kh^T:
//   P = exp(s - LSE),  dV = P^T dO,  dP = dO Vt^T,  Dlt = rowsum(dO * O),  dS = P * (dP - Dlt),
//   dQ = scale * dS Kh,  dK = scale * dS^T Qh;  a KV head's dK, dV sum over its query heads.
//
// Two kernels, 256 threads (8 warps) each, one CTA per SM:
//   * dK/dV: one CTA per (batch, KV head, 128-key tile); loops over the group's query heads and
//     the query tiles at or after the key tile, accumulating dV and dK in tensor memory;
//   * dQ: one CTA per (batch, query head, 128-row query tile); loops over the key tiles up to the
//     diagonal, accumulating dQ in tensor memory.
// S = Qh Kh^T is one block-scaled E4M3 MMA on the MXFP8 bytes and scales (exact products); dP, dV,
// dK and dQ are BF16 MMAs.  Every tile sits in shared memory in its natural orientation
// ([row][column], 64-column blocks with the 128-byte swizzle); the products that contract over
// its rows (P^T dO, dS^T Q, dS K) read it as an MN-major operand, so nothing is transposed.  In
// the dQ kernel the query tile's Q bytes and dO, and each iteration's dS, are the A operands of
// their MMAs from tensor memory.  The next iteration's copies are issued while the current one
// computes; the phases of an iteration run in turn, all threads taking part, thread 0 issuing the
// copies and MMAs.  Every wait is bounded.
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
constexpr int kThreads = 256;
constexpr uint32_t ATOM = 128 * 128;   // one 128-row x 128-byte swizzle block (64 BF16 columns)
// dS in tensor memory (64 BF16 columns over S) and its K order (ds_key_row) cover one 128-key tile
// in 16-key groups; the dQ MMA's K is that tile, its N the head dimension.
static_assert(BN == 128 && HD == 128, "tile shapes assumed by the tensor-memory layouts");

// TMEM columns: S, dP and two accumulators.  In the dK/dV kernel the scale factors of the S MMA
// sit at the start of dP's columns; dP is issued only once the S MMA has completed.
constexpr uint32_t T_S = 0, T_DP = 128, T_ACC0 = 256, T_ACC1 = 384;
// In the dQ kernel the query tile's operands stay in tensor memory: Q bytes (32 columns) and dO
// (BF16, 64 columns), the A operands of the S and dP MMAs.
constexpr uint32_t T_QT = 400, T_DOT = 432;

enum Site : int {
  W_KV = 0x20, W_QD, W_MMA1, W_MMA2, W_MMA3, W_DO, W_TMEM_BASE, W_PROD_S, W_PROD_QR, W_PROD_DK, W_DEC_KV, W_DEC_Q,
  W_DEC_DK, W_SM_DO, W_SM_S, W_SM_DP,
};

// A wait's outcome made the same for every thread of the CTA (the TMEM loads are warp-collective).
__device__ __forceinline__ bool cta_all(bool ok) { return __syncthreads_and(ok ? 1 : 0) != 0; }

// Byte offset of (row, byte column) inside a tile with 128-byte rows, 128-byte swizzle.
__device__ __forceinline__ uint32_t sw(uint32_t row, uint32_t colb) {
  return row * 128u + ((((colb >> 4) ^ row) & 7u) << 4) + (colb & 15u);
}
// Byte offset of BF16 element (row, col) of a 128 x 128 tile (two 64-column blocks).
__device__ __forceinline__ uint32_t bf_off(uint32_t row, uint32_t col) {
  return (col >> 6) * ATOM + sw(row, (col & 63u) * 2u);
}
__device__ __forceinline__ float pow2_e8m0(uint32_t sb) {
  return sb == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(sb << 23);   // 2^(sb-127)
}
// Compact rowwise scales of a 128-row tile (one 32-bit word per row, byte c for the 32-element
// block c) -> the tensor-core scale-factor atom: row m's word at (m % 32) * 16 + (m / 32) * 4.
// Rows at or past `nrows` get 0.  One warp; lane l writes the atom's 16-byte line l.
__device__ __forceinline__ void rows_to_atom(const uint8_t* compact, uint8_t* atom, int nrows, int lane) {
  const uint32_t* src = reinterpret_cast<const uint32_t*>(compact);
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] = lane + 32 * k < nrows ? src[lane + 32 * k] : 0u;
  *reinterpret_cast<uint4*>(atom + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
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

// E4M3 tile [row][d] (TMA, 128-byte swizzle) with compact row scales -> BF16 [row][d].  Rows at
// or past `nrows` become 0.
// Row position of key r in a decoded K tile that dQ's MMA reads against dS held in tensor memory:
// inside each 16-key group, key 8b + 2a + e (a < 4, b, e < 2) goes to row 4a + 2b + e, the K order
// of dS written with the 16x256b store (see dq_store_ds).
__device__ __forceinline__ int ds_key_row(int r) {
  return (r & ~15) | (((r >> 1) & 3) << 2) | (((r >> 3) & 1) << 1) | (r & 1);
}
template <bool PERM = false>
__device__ __forceinline__ void decode_rows(const uint8_t* src8, const uint8_t* sc_rows, uint8_t* dst, int nrows) {
  constexpr int kUnits = BM * (HD / 8) / kThreads;   // 8-element units per thread
  uint2 bytes[kUnits];
  float sc[kUnits];
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {   // every load first
    const int unit = threadIdx.x + u * kThreads, r = unit >> 4, d0 = (unit & 15) * 8;
    bytes[u] = *reinterpret_cast<const uint2*>(src8 + sw(r, d0));
    sc[u] = r < nrows ? pow2_e8m0(sc_rows[r * 4 + (d0 >> 5)]) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    const int unit = threadIdx.x + u * kThreads, r = unit >> 4, d0 = (unit & 15) * 8;
    *reinterpret_cast<uint4*>(dst + bf_off(PERM ? ds_key_row(r) : r, d0)) = decode8(bytes[u], sc[u]);
  }
}
// Token-normalised V bytes [key][d] (TMA, no swizzle) with one amplitude per key -> BF16 [key][d].
// Keys at or past `nkeys` become 0.
__device__ __forceinline__ void decode_vt(const uint8_t* raw, const uint8_t* amp, uint8_t* dst, int nkeys) {
  constexpr int kUnits = BN * (HD / 8) / kThreads;
  uint2 bytes[kUnits];
  float sc[kUnits];
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {   // every load first
    const int unit = threadIdx.x + u * kThreads, key = unit >> 4, d0 = (unit & 15) * 8;
    bytes[u] = *reinterpret_cast<const uint2*>(raw + key * HD + d0);
    sc[u] = key < nkeys ? pow2_e8m0(amp[key]) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    const int unit = threadIdx.x + u * kThreads, key = unit >> 4, d0 = (unit & 15) * 8;
    *reinterpret_cast<uint4*>(dst + bf_off(key, d0)) = decode8(bytes[u], sc[u]);
  }
}

// D (+)= A B^T over a 128-deep contraction in eight BF16 MMAs of K = 16.  A tile read along its
// columns (K-major) advances 32 bytes per step inside a block; one read along its rows (MN-major,
// idesc bit 15 for A, 16 for B) advances 16 rows = 2048 bytes, with its two 64-column blocks
// 16 KB apart.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma_bf16_k128(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, bool accumulate) {
  const uint32_t idesc = idesc_bf16(BM, BN) | (A_MN ? (1u << 15) : 0u) | (B_MN ? (1u << 16) : 0u);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint64_t da = A_MN ? smem_desc(a_smem + s * 2048, ATOM, 1024, 2)
                             : desc_kmajor_sw128(a_smem + (s >> 2) * ATOM + (s & 3) * 32);
    const uint64_t db = B_MN ? smem_desc(b_smem + s * 2048, ATOM, 1024, 2)
                             : desc_kmajor_sw128(b_smem + (s >> 2) * ATOM + (s & 3) * 32);
    mma_f16_ss(d_tmem, da, db, idesc, (accumulate || s > 0) ? 1u : 0u);
  }
}
// S = Qh Kh^T with the Q bytes in tensor memory (columns t_q..t_q+31).
__device__ __forceinline__ void mma_s_tq(uint32_t tmem, uint32_t t_sf, uint32_t t_q, uint32_t k8, uint32_t sfq,
                                         uint32_t sfk) {
  tc_cp_32x128b_warpx4(tmem + t_sf, desc_sf_block(sfq));
  tc_cp_32x128b_warpx4(tmem + t_sf + 4, desc_sf_block(sfk));
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    mma_mxf8_ts(tmem + T_S, tmem + t_q + 8 * kk, desc_kmajor_sw128(k8 + kk * 32), idesc_mxf8(BM, BN, kk, kk),
                tmem + t_sf, tmem + t_sf + 4, kk > 0 ? 1u : 0u);
  }
}

// One thread's view of a 16x256b TMEM load: rows ra = base + lane/4 and rb = ra + 8, keys
// 8k + 2(lane%4) + e at v[4k + e] (row ra) and v[4k + 2 + e] (row rb).
struct RowView {
  int base, ra, rb, qd;
  uint32_t lane_off;
};
__device__ __forceinline__ RowView row_view() {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  RowView v;
  v.base = (warp & 3) * 32 + (warp >> 2) * 16;
  v.ra = v.base + (lane >> 2);
  v.rb = v.ra + 8;
  v.qd = lane & 3;
  v.lane_off = (uint32_t)v.base << 16;
  return v;
}

// P = exp(s - LSE) of this thread's 64 elements from S in TMEM; in the diagonal tile keys after
// the row are masked.
__device__ __forceinline__ void compute_p(uint32_t tmem, const RowView& rv, const float* lse2, float sl2, bool diag,
                                          float (&p)[64]) {
  tmem_ld16x256_x16(tmem + T_S + rv.lane_off, p);
  tmem_ld_wait();
  const float la = lse2[rv.ra], lb = lse2[rv.rb];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = 8 * k + 2 * rv.qd + e;
      p[4 * k + e] = (diag && key > rv.ra) ? 0.f : ex2_approx(fmaf(p[4 * k + e], sl2, -la));
      p[4 * k + 2 + e] = (diag && key > rv.rb) ? 0.f : ex2_approx(fmaf(p[4 * k + 2 + e], sl2, -lb));
    }
  }
}
// dS = P (dP - Dlt) from dP in TMEM.
__device__ __forceinline__ void compute_ds(uint32_t tmem, const RowView& rv, const float* dlt, const float (&p)[64],
                                           float (&ds)[64]) {
  tmem_ld16x256_x16(tmem + T_DP + rv.lane_off, ds);
  tmem_ld_wait();
  const float da = dlt[rv.ra], db = dlt[rv.rb];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      ds[4 * k + e] = p[4 * k + e] * (ds[4 * k + e] - da);
      ds[4 * k + 2 + e] = p[4 * k + 2 + e] * (ds[4 * k + 2 + e] - db);
    }
  }
}
// dS as BF16 into tensor memory (64 columns from t_ds), the A operand of dQ += dS K: register
// 4c + 2rr + b of the 16x256b store (row ra or rb for rr = 0, 1; column 8c + 2qd + b) holds the
// keys 16c + 8b + 2qd and the next, so column 8c + 2qd + b carries K positions 16c + 4qd + 2b + e
// for keys 16c + 8b + 2qd + e; the decoded K tile's rows use the same order (ds_key_row).
__device__ __forceinline__ void dq_store_ds(uint32_t t_ds, const RowView& rv, const float (&ds)[64]) {
  uint32_t w[32];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int k = 2 * c + b;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) w[4 * c + 2 * rr + b] = pack_bf16x2(ds[4 * k + 2 * rr], ds[4 * k + 2 * rr + 1]);
    }
  }
  tmem_st16x256_x8(t_ds + rv.lane_off, w);
}

// Epilogue: an accumulator (128 rows x 128 columns fp32 in TMEM) times `mul` -> BF16 rows of a
// tensor laid out like Q (BSHD/SBHD with H heads); rows at or past S are not written.
__device__ __forceinline__ void store_acc(uint32_t tmem_acc, void* out, const BwdArgs& a, int H, int b, int h,
                                          int tile, float mul) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qq = warp & 3, half = warp >> 2;
  const int r = qq * 32 + lane;
  const int i = tile * BM + r;
  float o[2][32];
  const uint32_t ta = tmem_acc + ((uint32_t)(qq * 32) << 16) + 64 * half;
  tmem_ld32f(ta, o[0]);
  tmem_ld32f(ta + 32, o[1]);
  tmem_ld_wait();
  if (i >= a.S) return;
  const long long row = a.layout == 0 ? ((long long)b * a.S + i) * H + h : ((long long)i * a.B + b) * H + h;
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + row * HD + 64 * half);
#pragma unroll
  for (int e8 = 0; e8 < 8; ++e8) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = e8 * 8 + 2 * e;
      w[e] = pack_bf16x2(o[k >> 5][k & 31] * mul, o[(k + 1) >> 5][(k + 1) & 31] * mul);
    }
    dst[e8] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ================================================================================================
// Row statistics of the backward, once per call: Dlt_i = <dO_i, O_i> and LSE_i * log2(e) of every
// query row into the workspace, two planes [B][Hq][Sp] of fp32 (Sp = 128 * ceil(S / 128)).  Rows
// at or past S get Dlt = 0 and +inf, which make their P and dS exactly 0.  One warp per row.
__global__ void __launch_bounds__(256) attn_bwd_stats_kernel(const __grid_constant__ BwdArgs a) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)a.B * a.Hq * a.Sp;
  const long long rid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (rid >= rows) return;
  const int i = (int)(rid % a.Sp);
  const long long bh = rid / a.Sp;
  const int hq = (int)(bh % a.Hq), b = (int)(bh / a.Hq);
  float acc = 0.f;
  if (i < a.S) {
    const long long row = a.layout == 0 ? ((long long)b * a.S + i) * a.Hq + hq : ((long long)i * a.B + b) * a.Hq + hq;
    const uint2 x = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.o) + row * HD) + lane);
    const uint2 y = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.dO) + row * HD) + lane);
    const uint32_t xs[2] = {x.x, x.y}, ys[2] = {y.x, y.y};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      acc = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), acc);
      acc = fmaf(__uint_as_float(xs[e] & 0xFFFF0000u), __uint_as_float(ys[e] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) {
    a.ws[rid] = i < a.S ? acc : 0.f;
    a.ws[rows + rid] = i < a.S ? a.lse[bh * a.S + i] * 1.4426950408889634f : INFINITY;
  }
}

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
// Eight E4M3 bytes (one uint2, element e in byte e) times scale2 (BF16x2) -> eight BF16 (one uint4).
__device__ __forceinline__ uint4 decode8_bf16(uint2 bytes, uint32_t scale2) {
  constexpr uint32_t kTwo120 = 0x7B807B80u;   // 2^120 in both halves
  uint32_t w[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t x = h ? bytes.y : bytes.x;
    w[2 * h] = bf16x2_mul(bf16x2_mul(e4m3x2_times_2m120(__byte_perm(x, 0u, 0x4140)), kTwo120), scale2);
    w[2 * h + 1] = bf16x2_mul(bf16x2_mul(e4m3x2_times_2m120(__byte_perm(x, 0u, 0x4342)), kTwo120), scale2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// A 128 x 128 E4M3 tile -> BF16 [row][d] (two 64-column blocks, 128-byte swizzle) by `nthr`
// threads (index t).  Source rows are 128 bytes, swizzled (SW = true, as TMA writes a Q or K tile)
// or plain (the token-normalised V tile); scale of (row r, 32-element block c) is
// row_scale(r, c).  Each thread keeps one 8-element column position and walks rows nthr/16 apart.
template <bool SW, int NTHR, typename RowScale>
__device__ __forceinline__ void decode_tile_bf16(const uint8_t* src, uint8_t* dst, int t, RowScale row_scale) {
  constexpr int kUnits = BM * (HD / 8) / NTHR;   // eight-element units per thread
  constexpr int kBatch = 16;
  static_assert(kUnits % kBatch == 0, "batches");
  const int d0 = (t & 15) * 8, r0 = t >> 4;
#pragma unroll 1
  for (int u0 = 0; u0 < kUnits; u0 += kBatch) {
    uint2 bytes[kBatch];
    uint32_t sc[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {   // every load of the batch first
      const int r = r0 + (NTHR / 16) * (u0 + u);
      bytes[u] = *reinterpret_cast<const uint2*>(src + (SW ? sw(r, d0) : (uint32_t)(r * HD + d0)));
      sc[u] = row_scale(r, d0 >> 5);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = r0 + (NTHR / 16) * (u0 + u);
      *reinterpret_cast<uint4*>(dst + bf_off(r, d0)) = decode8_bf16(bytes[u], sc[u]);
    }
  }
}

// ================================================================================================
// dK, dV.  One CTA per (batch, KV head, 128-key tile jt); it walks the pairs n = 0..N-1 of (query
// head of the group, query tile at or after jt): query tiles from the last down, the group's heads
// innermost, so that CTAs of one KV head running at the same time read the same Q and dO tiles from
// L2.  The keys sit on the TMEM lanes, so P^T and dS^T are the A operands of the dV and dK MMAs
// straight from tensor memory:
//   S^T  = Kh Qh^T      block-scaled E4M3 MMA on the bytes (A = K, B = Q, both K-major)
//   dP^T = Vt dO^T      BF16 (A = Vt [key][d], B = dO [q][d], both K-major)
//   P^T  = exp2(S^T scale log2(e) - LSE2[q]),  dS^T = P^T (dP^T - Dlt[q])     (softmax warps)
//   dV  += P^T dO       A = P^T (BF16 over the first 64 columns of S^T), B = dO read along q
//   dK  += dS^T Qh      A = dS^T (BF16 over the first 64 columns of dP^T), B = decoded Q along q
// Roles (8 warps): warp 0 lane 0 issues the copies; warp 1 lane 0 issues the MMAs in the order
//   S(0) dP(0) | dV(n) S(n+1) dK(n) dP(n+1) | ...
// so that the softmax of pair n + 1 runs under dK(n) and dP(n + 1); warps 2-3 decode (V once, the Q
// bytes of every pair to BF16, the scale atoms); warps 4-7 compute P and dS, one key row per
// thread.  TMEM: S^T 0-127, dP^T 128-255, dV 256-383, dK 384-511.  The S MMA's scale factors sit in
// dP^T's columns 120-127: the softmax reads those columns of dP^T(n) before it releases P(n), after
// which S(n + 1) is issued.  An MMA that rewrites columns an earlier one reads (S(n+1) over P^T(n),
// dP(n+1) over dS^T(n) and the scale factors) is issued after it: the MMAs of one thread run in
// issue order.  The MMA-issuing thread waits on named barriers only (an mbarrier wait there drains
// its MMAs in flight).
//
// Shared memory (bytes from a 1024-aligned base):
constexpr uint32_t KV_K8 = 0;                    // K bytes [key][d], swizzled
constexpr uint32_t KV_V = KV_K8 + 16384;         // V bf16 [key][d]
constexpr uint32_t KV_Q8 = KV_V + 32768;         // 2 stages: Q bytes [q][d], swizzled
constexpr uint32_t KV_Q = KV_Q8 + 2 * 16384;     // 2 stages: decoded Q bf16 [q][d]
constexpr uint32_t KV_VN8 = KV_Q + 32768;        // V bytes [key][d], in Q stage 1 before its first use
constexpr uint32_t KV_DO = KV_Q + 2 * 32768;     // 2 stages: dO bf16 [q][d]
constexpr uint32_t KV_SFQ = KV_DO + 2 * 32768;   // 2 stages: compact Q scales
constexpr uint32_t KV_SFK = KV_SFQ + 1024;       // compact K scales
constexpr uint32_t KV_SFQA = KV_SFK + 512;       // 2 stages: Q scale atoms
constexpr uint32_t KV_SFKA = KV_SFQA + 1024;     // K scale atom
constexpr uint32_t KV_AMP = KV_SFKA + 512;       // V token amplitudes
constexpr uint32_t KV_STAT = KV_AMP + 128;       // 2 stages: Dlt[128], then LSE2[128]
constexpr uint32_t KV_BAR = KV_STAT + 2048;
constexpr uint32_t KV_MISC = KV_BAR + 128;       // TMEM slot, abort flag
constexpr uint32_t KV_SMEM = KV_MISC + 16 + 1024;
static_assert(KV_SMEM <= 227 * 1024, "shared memory budget");
constexpr uint32_t T_ST = 0, T_DPT = 128, T_DV = 256, T_DK = 384;
constexpr uint32_t T_SFK = T_DPT + 120, T_SFQ = T_DPT + 124;
// mbarriers:
//   KV         K, its scales, the V bytes and amplitudes landed
//   QF + st    Q bytes and compact scales of stage st landed
//   DF + st    dO and the row statistics of stage st landed
//   SF + n%2   S^T(n) computed (and every MMA issued before it)
//   DP         dP^T(n) computed
//   DK + n%2   dK(n) computed (and every MMA issued before it)
//   QR + st    the decoders are done with Q stage st (count 2: one arrival per decoder warp)
enum KvBar : uint32_t {
  KB_KV = 0,
  KB_QF = 1,
  KB_DF = KB_QF + 2,
  KB_SF = KB_DF + 2,
  KB_DP = KB_SF + 2,
  KB_DK,
  KB_QR = KB_DK + 2,
  KB_DRAIN = KB_QR + 2,
  KB_COUNT
};
static_assert(KB_COUNT * 8 <= 128, "barrier slots");
// Named barriers (each with the MMA warp):
//   NB_KV        decoders: the K scale atom and the BF16 V tile are written (once)
//   NB_Q + n%2   decoders: the Q scale atom of pair n is written
//   NB_QD + n%2  decoders: the BF16 Q of pair n is written
//   NB_DO        softmax: dO of pair n landed
//   NB_P         softmax: P^T(n) is in TMEM, and columns 96-127 of dP^T(n) are read
//   NB_DS        softmax: dS^T(n) is in TMEM
// The decoders block on NB_QD and the softmax warps on NB_DS, and arrive on the others: each
// blocking generation they pass shows the MMA warp has passed the previous generation of every
// barrier they arrive on next, so no generation ever holds arrivals of two pairs, also once a role
// has given up (failed wait: it skips its work but meets every generation).  Both meet their
// generations in the MMA warp's order (the decoders Q(n+1) before QD(n)), so none waits forever.
constexpr uint32_t NB_KV = 1, NB_Q = 2, NB_QD = 4, NB_DO = 6, NB_P = 7, NB_DS = 8, NB_DEC = 9;
constexpr uint32_t kNbDec = 96, kNbSm = 160;

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
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
  const int bh = blockIdx.x % (a.B * a.Hkv);
  const int jt = (int)(blockIdx.x / (a.B * a.Hkv));
  const int hk = bh % a.Hkv, b = bh / a.Hkv;
  const long long kv_plane = (long long)b * a.Hkv + hk;
  const int nkeys = min(BN, a.S - jt * BN);
  const int N = g * (T - jt);   // pairs; the last g of them are the diagonal tile
  auto hq_of = [&](int n) { return hk * g + n % g; };
  auto it_of = [&](int n) { return T - 1 - n / g; };

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < KB_COUNT; ++i) mbar_init(bar(i), (i == KB_QR || i == KB_QR + 1) ? 2u : 1u);
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
      prefetch_tensormap(&a.tm_q);
      prefetch_tensormap(&a.tm_k);
      prefetch_tensormap(&a.tm_vtn);
      prefetch_tensormap(&a.tm_do);
      const long long ws_plane = (long long)a.B * a.Hq * a.Sp;
      auto load_q = [&](int n) {
        const int st = n & 1, it = it_of(n), hq = hq_of(n);
        const uint32_t nr = (uint32_t)min(BM, a.S - it * BM);
        mbar_arrive_expect_tx(bar(KB_QF + st), BM * HD + 4 * nr);
        tma_load_4d(sbase + KV_Q8 + st * 16384, &a.tm_q, bar(KB_QF + st), 0, hq, it * BM, b);
        bulk_load(sbase + KV_SFQ + st * 512, a.q_sc + (((long long)b * a.Hq + hq) * a.S + (long long)it * BM) * 4,
                  4 * nr, bar(KB_QF + st));
      };
      auto load_do = [&](int n) {
        const int st = n & 1, it = it_of(n), hq = hq_of(n);
        const long long srow = ((long long)b * a.Hq + hq) * a.Sp + (long long)it * BM;
        mbar_arrive_expect_tx(bar(KB_DF + st), 2 * BM * HD + 1024);
        tma_load_4d(sbase + KV_DO + st * 32768, &a.tm_do, bar(KB_DF + st), 0, hq, it * BM, b);
        tma_load_4d(sbase + KV_DO + st * 32768 + ATOM, &a.tm_do, bar(KB_DF + st), 64, hq, it * BM, b);
        bulk_load(sbase + KV_STAT + st * 1024, a.ws + srow, 512, bar(KB_DF + st));
        bulk_load(sbase + KV_STAT + st * 1024 + 512, a.ws + ws_plane + srow, 512, bar(KB_DF + st));
      };
      bool ok = start_ok;
      int nq[2] = {0, 0}, nd[2] = {0, 0};
      if (ok) {
        mbar_arrive_expect_tx(bar(KB_KV), 2 * BN * HD + 4 * (uint32_t)nkeys + (uint32_t)nkeys);
        tma_load_4d(sbase + KV_K8, &a.tm_k, bar(KB_KV), 0, hk, jt * BN, b);
        bulk_load(sbase + KV_SFK, a.k_sc + (kv_plane * a.S + (long long)jt * BN) * 4, 4 * (uint32_t)nkeys,
                  bar(KB_KV));
        tma_load_4d(sbase + KV_VN8, &a.tm_vtn, bar(KB_KV), 0, hk, jt * BN, b);
        bulk_load(sbase + KV_AMP, a.vtn_sc + kv_plane * a.S + (long long)jt * BN, (uint32_t)nkeys, bar(KB_KV));
        for (int n = 0; n < 2 && n < N; ++n) {
          load_q(n);
          load_do(n);
          nq[n] = nd[n] = 1;
        }
      }
      // Stage n % 2 takes pair n + 2 once pair n is done with it: the Q bytes after S^T(n) and the
      // decode of Q(n); dO and the statistics after dK(n) (the softmax has used them by then).
      for (int n = 0; ok && n + 2 < N; ++n) {
        const int st = n & 1;
        const uint32_t ph = (uint32_t)(n >> 1) & 1u;
        if (!(ok = mbar_wait(bar(KB_SF + st), ph, ctl, W_PROD_S))) break;
        if (!(ok = mbar_wait(bar(KB_QR + st), ph, ctl, W_PROD_QR))) break;
        load_q(n + 2);
        ++nq[st];
        if (!(ok = mbar_wait(bar(KB_DK + st), ph, ctl, W_PROD_DK))) break;
        load_do(n + 2);
        ++nd[st];
      }
      // every copy this thread issued lands before the CTA may exit
      if (start_ok) mbar_wait_drain(bar(KB_KV), 0, a.limit_ns);
      for (int st = 0; st < 2; ++st) {
        if (nq[st] > 0) mbar_wait_drain(bar(KB_QF + st), (uint32_t)(nq[st] - 1) & 1u, a.limit_ns);
        if (nd[st] > 0) mbar_wait_drain(bar(KB_DF + st), (uint32_t)(nd[st] - 1) & 1u, a.limit_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer: lane 0 issues, the whole warp meets the named barriers
    const bool ok = start_ok;
    auto live = [&]() { return ok && *abort_flag == 0; };
    const uint64_t dK8 = desc_kmajor_sw128(sbase + KV_K8), dQ8 = desc_kmajor_sw128(sbase + KV_Q8);
    const uint64_t dVk = desc_kmajor_sw128(sbase + KV_V), dDOk = desc_kmajor_sw128(sbase + KV_DO);
    const uint64_t dDOm = smem_desc(sbase + KV_DO, ATOM, 1024, 2), dQm = smem_desc(sbase + KV_Q, ATOM, 1024, 2);
    constexpr uint32_t idS = idesc_mxf8(BN, BM, 0, 0);
    constexpr uint32_t idP = idesc_bf16(BN, BM), idMN = idesc_bf16(BN, HD) | (1u << 16);
    auto issue_s = [&](int n) {   // S^T = K Q^T (block-scaled)
      const uint32_t st = (uint32_t)n & 1u;
      tc_cp_32x128b_warpx4(tmem + T_SFK, desc_sf_block(sbase + KV_SFKA));
      tc_cp_32x128b_warpx4(tmem + T_SFQ, desc_sf_block(sbase + KV_SFQA + 512 * st));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_mxf8_ss(tmem + T_ST, dK8 + 2 * kk, dQ8 + st * (16384 >> 4) + 2 * kk,
                    idS | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), tmem + T_SFK, tmem + T_SFQ, kk > 0 ? 1u : 0u);
      }
      tc_commit(bar(KB_SF + st));
    };
    auto issue_dp = [&](int n) {  // dP^T = V dO^T
      const uint64_t db = dDOk + ((uint32_t)n & 1u) * (32768 >> 4);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t off = ((s >> 2) * ATOM + (s & 3) * 32) >> 4;
        mma_f16_ss(tmem + T_DPT, dVk + off, db + off, idP, s > 0 ? 1u : 0u);
      }
      tc_commit(bar(KB_DP));
    };
    auto issue_dv = [&](int n) {  // dV += P^T dO
      const uint64_t db = dDOm + ((uint32_t)n & 1u) * (32768 >> 4);
      const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
      for (int s = 0; s < 8; ++s) mma_f16_ts(tmem + T_DV, tmem + T_ST + 8 * s, db + s * (2048 >> 4), idMN, s > 0 ? 1u : acc0);
    };
    auto issue_dk = [&](int n) {  // dK += dS^T Q
      const uint64_t db = dQm + ((uint32_t)n & 1u) * (32768 >> 4);
      const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
      for (int s = 0; s < 8; ++s) mma_f16_ts(tmem + T_DK, tmem + T_DPT + 8 * s, db + s * (2048 >> 4), idMN, s > 0 ? 1u : acc0);
      tc_commit(bar(KB_DK + ((uint32_t)n & 1u)));
    };
    named_sync(NB_KV, kNbDec);
    named_sync(NB_Q + 0, kNbDec);
    if (lane == 0 && live()) {
      tc_fence_after();
      issue_s(0);
    }
    __syncwarp();
    named_sync(NB_DO, kNbSm);
    if (lane == 0 && live()) {
      tc_fence_after();
      issue_dp(0);
    }
    __syncwarp();
    for (int n = 0; n < N; ++n) {
      named_sync(NB_P, kNbSm);
      if (lane == 0 && live()) {
        tc_fence_after();
        issue_dv(n);
      }
      __syncwarp();
      if (n + 1 < N) {
        named_sync(NB_Q + ((n + 1) & 1), kNbDec);
        if (lane == 0 && live()) {
          tc_fence_after();
          issue_s(n + 1);
        }
        __syncwarp();
      }
      named_sync(NB_QD + (n & 1), kNbDec);
      named_sync(NB_DS, kNbSm);
      if (lane == 0 && live()) {
        tc_fence_after();
        issue_dk(n);
      }
      __syncwarp();
      if (n + 1 < N) {
        named_sync(NB_DO, kNbSm);
        if (lane == 0 && live()) {
          tc_fence_after();
          issue_dp(n + 1);
        }
        __syncwarp();
      }
    }
    if (lane == 0) tc_commit(bar(KB_DRAIN));   // every MMA of the CTA
    __syncwarp();
  } else if (warp < 4) {
    // ======================= decoders (64 threads): the K scale atom and BF16 V once, then per
    // pair the Q scale atom (one pair ahead) and the BF16 Q
    const int t = threadIdx.x - 64;
    bool ok = start_ok && __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_KV), 0, ctl, W_DEC_KV));
    if (ok) {
      if (warp == 2) rows_to_atom(smem + KV_SFK, smem + KV_SFKA, nkeys, lane);
      const uint8_t* amp = smem + KV_AMP;
      decode_tile_bf16<false, 64>(smem + KV_VN8, smem + KV_V, t, [&](int r, int) {
        return r < nkeys ? bf16x2_pow2_e8m0(amp[r]) : 0u;
      });
    }
    fence_proxy_async_smem();
    named_sync(NB_DEC, 64);   // every V byte is read before Q stage 1 is written
    named_arrive(NB_KV, kNbDec);
    auto atom = [&](int n) {   // the Q scale atom of pair n, once its copy landed
      const int st = n & 1;
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_QF + st), (uint32_t)(n >> 1) & 1u, ctl, W_DEC_Q));
      if (ok && warp == 2) rows_to_atom(smem + KV_SFQ + st * 512, smem + KV_SFQA + st * 512, min(BM, a.S - it_of(n) * BM), lane);
      fence_proxy_async_smem();
      named_arrive(NB_Q + st, kNbDec);
    };
    atom(0);
    for (int n = 0; n < N; ++n) {
      const int st = n & 1;
      if (n + 1 < N) atom(n + 1);
      // Q stage st in BF16, once dK(n - 2), its last reader, has completed
      if (n >= 2 && ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_DK + st), (uint32_t)((n - 2) >> 1) & 1u, ctl, W_DEC_DK));
      if (ok) {
        const int nr = min(BM, a.S - it_of(n) * BM);
        const uint8_t* sfq = smem + KV_SFQ + st * 512;
        decode_tile_bf16<true, 64>(smem + KV_Q8 + st * 16384, smem + KV_Q + st * 32768, t, [&](int r, int c) {
          return r < nr ? bf16x2_pow2_e8m0(sfq[r * 4 + c]) : 0u;
        });
      }
      fence_proxy_async_smem();
      named_sync(NB_QD + st, kNbDec);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KB_QR + st));
    }
  } else {
    // ======================= softmax: key row kr of the tile per thread
    const int qq = warp & 3, kr = qq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const float sl2 = a.scale_log2e;
    bool ok = start_ok;
    // dS of 32 queries from their P, dP and Dlt, packed to BF16 pairs
    auto ds_chunk = [&](const float* p, const float* d, const float* dlt, uint32_t* w) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 dl = *reinterpret_cast<const float2*>(dlt + 2 * i);
        w[i] = pack_bf16x2(p[2 * i] * (d[2 * i] - dl.x), p[2 * i + 1] * (d[2 * i + 1] - dl.y));
      }
    };
    auto pair = [&](int n, auto diag_tag) {
      constexpr bool DIAG = decltype(diag_tag)::value;
      const int st = n & 1;
      const float* dlt = reinterpret_cast<const float*>(smem + KV_STAT + st * 1024);
      const float* lse2 = dlt + 128;
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_DF + st), (uint32_t)(n >> 1) & 1u, ctl, W_SM_DO));
      named_arrive(NB_DO, kNbSm);
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_SF + st), (uint32_t)(n >> 1) & 1u, ctl, W_SM_S));
      float p[128];
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) tld32(tmem + lane_off + T_ST + 32 * c, p + 32 * c);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 32; ++q4) {
          const float4 l = *reinterpret_cast<const float4*>(lse2 + 4 * q4);
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = 4 * q4 + e;
            const float x = ex2_approx(fmaf(p[q], sl2, -lv[e]));
            p[q] = (DIAG && q < kr) ? 0.f : x;   // in the diagonal tile a query sees keys up to itself
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(p[32 * c + 2 * i], p[32 * c + 2 * i + 1]);
          tst16(tmem + lane_off + T_ST + 16 * c, w);
        }
      }
      uint32_t ds3[16];
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(KB_DP), (uint32_t)n & 1u, ctl, W_SM_DP));
      if (ok) {
        tc_fence_after();
        float d[32];
        tld32(tmem + lane_off + T_DPT + 96, d);   // the columns the next S MMA's scales go into
        tmem_ld_wait();
        ds_chunk(p + 96, d, dlt + 96, ds3);
        tmem_st_wait();
        tc_fence_before();
      }
      named_arrive(NB_P, kNbSm);
      if (ok) {
        // dS^T of queries 32c.. goes over columns 16c.., which hold dP^T of queries read by then
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          float d[32];
          uint32_t w[16];
          tld32(tmem + lane_off + T_DPT + 32 * c, d);
          tmem_ld_wait();
          ds_chunk(p + 32 * c, d, dlt + 32 * c, w);
          tst16(tmem + lane_off + T_DPT + 16 * c, w);
          if (c == 1) tst16(tmem + lane_off + T_DPT + 48, ds3);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      named_sync(NB_DS, kNbSm);
    };
    int n = 0;
    for (; n < N - g; ++n) pair(n, std::false_type{});
    for (; n < N; ++n) pair(n, std::true_type{});
  }

  // ======================= epilogue: dV and dK from TMEM, 8 warps
  tc_fence_before();
  __syncthreads();
  const bool drained = mbar_wait_drain(bar(KB_DRAIN), 0, a.limit_ns);
  tc_fence_after();
  if (cta_all(drained && start_ok && *abort_flag == 0)) {
    store_acc(tmem + T_DV, a.dv, a, a.Hkv, b, hk, jt, 1.0f);
    store_acc(tmem + T_DK, a.dk, a, a.Hkv, b, hk, jt, a.scale);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ================================================================================================
// dQ.  Shared memory:
constexpr uint32_t QQ_Q8 = 0;                       // Q bytes [q][d], swizzled
constexpr uint32_t QQ_DO = QQ_Q8 + 16384;           // dO bf16 [q][d]
constexpr uint32_t QQ_K8 = QQ_DO + 32768;           // 2 stages: K bytes [key][d], swizzled
constexpr uint32_t QQ_VN8 = QQ_K8 + 2 * 16384;      // 2 stages: token-normalised V bytes [key][d]
constexpr uint32_t QQ_K = QQ_VN8 + 2 * 16384;       // K bf16 [key][d], rows in the order of ds_key_row
constexpr uint32_t QQ_V = QQ_K + 32768;             // V bf16 [key][d]
constexpr uint32_t QQ_SFQ = QQ_V + 32768;           // compact Q scales of the tile
constexpr uint32_t QQ_SFK = QQ_SFQ + 512;           // 2 stages of compact K scales
constexpr uint32_t QQ_SFQA = QQ_SFK + 1024;         // Q scale atom
constexpr uint32_t QQ_SFKA = QQ_SFQA + 512;         // K scale atom of the current key tile
constexpr uint32_t QQ_AMP = QQ_SFKA + 512;          // 2 stages of 128
constexpr uint32_t QQ_LSE = QQ_AMP + 256;
constexpr uint32_t QQ_DLT = QQ_LSE + 512;
constexpr uint32_t QQ_BAR = QQ_DLT + 512;
constexpr uint32_t QQ_MISC = QQ_BAR + 64;
constexpr uint32_t QQ_SMEM = QQ_MISC + 16 + 1024;
static_assert(QQ_SMEM <= 227 * 1024, "shared memory budget");
enum QBar : uint32_t { QB_QD = 0, QB_KV0, QB_KV1, QB_MMA1, QB_MMA2, QB_DRAIN, QB_COUNT };

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](uint32_t i) { return sbase + QQ_BAR + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + QQ_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + QQ_MISC + 4);
  float* lse2 = reinterpret_cast<float*>(smem + QQ_LSE);
  float* dlt = reinterpret_cast<float*>(smem + QQ_DLT);

  const int T = (a.S + BM - 1) / BM;
  const int bh = blockIdx.x % (a.B * a.Hq);
  const int it = T - 1 - (int)(blockIdx.x / (a.B * a.Hq));   // heaviest query tiles first
  const int hq = bh % a.Hq, b = bh / a.Hq;
  const int hk = hq / (a.Hq / a.Hkv);
  const long long kv_plane = (long long)b * a.Hkv + hk;

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < QB_COUNT; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(sbase + QQ_MISC, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, a.dev_status, a.limit_ns};
  const bool leader = threadIdx.x == 0;
  // key tile j into stage j % 2
  auto load_kv = [&](int j) {
    const int st = j & 1;
    const uint32_t nk = (uint32_t)min(BN, a.S - j * BN);
    const uint32_t kb = bar(QB_KV0 + st);
    mbar_arrive_expect_tx(kb, 2 * BN * HD + 4 * nk + nk);
    tma_load_4d(sbase + QQ_K8 + st * 16384, &a.tm_k, kb, 0, hk, j * BN, b);
    bulk_load(sbase + QQ_SFK + st * 512, a.k_sc + (kv_plane * a.S + (long long)j * BN) * 4, 4 * nk, kb);
    tma_load_4d(sbase + QQ_VN8 + st * 16384, &a.tm_vtn, kb, 0, hk, j * BN, b);
    bulk_load(sbase + QQ_AMP + st * 128, a.vtn_sc + kv_plane * a.S + (long long)j * BN, nk, kb);
  };
  bool ok = true;
  int kv_issued[2] = {0, 0}, kv_seen[2] = {0, 0};

  if (leader) {
    const uint32_t nr = (uint32_t)min(BM, a.S - it * BM);
    mbar_arrive_expect_tx(bar(QB_QD), BM * HD + 4 * nr + 2 * BM * HD);
    tma_load_4d(sbase + QQ_Q8, &a.tm_q, bar(QB_QD), 0, hq, it * BM, b);
    bulk_load(sbase + QQ_SFQ, a.q_sc + (((long long)b * a.Hq + hq) * a.S + (long long)it * BM) * 4, 4 * nr,
              bar(QB_QD));
    tma_load_4d(sbase + QQ_DO, &a.tm_do, bar(QB_QD), 0, hq, it * BM, b);
    tma_load_4d(sbase + QQ_DO + ATOM, &a.tm_do, bar(QB_QD), 64, hq, it * BM, b);
    load_kv(0);
  }
  kv_issued[0] = 1;
  if (threadIdx.x < BM) {   // the tile's row statistics, written by the statistics kernel
    const long long srow = ((long long)b * a.Hq + hq) * a.Sp + (long long)it * BM + threadIdx.x;
    dlt[threadIdx.x] = a.ws[srow];
    lse2[threadIdx.x] = a.ws[(long long)a.B * a.Hq * a.Sp + srow];
  }
  ok = cta_all(mbar_wait(bar(QB_QD), 0, ctl, W_QD));
  const bool qd_seen = ok;
  if (ok && threadIdx.x < 32) {
    rows_to_atom(smem + QQ_SFQ, smem + QQ_SFQA, min(BM, a.S - it * BM), threadIdx.x);
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (leader && ok) {   // the Q bytes and dO into tensor memory, once
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) tc_cp_128x256b(tmem + T_QT + 8 * kk, desc_kmajor_sw128(sbase + QQ_Q8 + kk * 32));
#pragma unroll
    for (int s = 0; s < 8; ++s)
      tc_cp_128x256b(tmem + T_DOT + 8 * s, desc_kmajor_sw128(sbase + QQ_DO + (s >> 2) * ATOM + (s & 3) * 32));
  }

  const RowView rv = row_view();
  for (int jt = 0; jt <= it; ++jt) {
    const uint32_t par = (uint32_t)jt & 1u;
    const int st = jt & 1;
    const int nkeys = min(BN, a.S - jt * BN);
    if (leader && ok && jt + 1 <= it) load_kv(jt + 1);   // stage st^1 was last read in iteration jt-1
    if (ok && jt + 1 <= it) ++kv_issued[st ^ 1];
    if (ok) ok = mbar_wait(bar(QB_KV0 + st), (uint32_t)(jt >> 1) & 1u, ctl, W_KV);
    ok = cta_all(ok);
    if (ok) ++kv_seen[st];
    if (ok) {
      if (threadIdx.x < 32) rows_to_atom(smem + QQ_SFK + st * 512, smem + QQ_SFKA, nkeys, threadIdx.x);
      decode_vt(smem + QQ_VN8 + st * 16384, smem + QQ_AMP + st * 128, smem + QQ_V, nkeys);
      decode_rows<true>(smem + QQ_K8 + st * 16384, smem + QQ_SFK + st * 512, smem + QQ_K, nkeys);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (leader && ok) {
      mma_s_tq(tmem, T_ACC1, T_QT, sbase + QQ_K8 + st * 16384, sbase + QQ_SFQA, sbase + QQ_SFKA);
#pragma unroll
      for (int s = 0; s < 8; ++s) {   // dP = dO V^T, dO from tensor memory
        mma_f16_ts(tmem + T_DP, tmem + T_DOT + 8 * s,
                   desc_kmajor_sw128(sbase + QQ_V + (s >> 2) * ATOM + (s & 3) * 32), idesc_bf16(BM, BN),
                   s > 0 ? 1u : 0u);
      }
      tc_commit(bar(QB_MMA1));
    }
    if (ok) ok = mbar_wait(bar(QB_MMA1), par, ctl, W_MMA1);
    ok = cta_all(ok);
    tc_fence_after();
    if (ok) {
      float p[64], ds[64];
      compute_p(tmem, rv, lse2, a.scale_log2e, jt == it, p);
      compute_ds(tmem, rv, dlt, p, ds);
      dq_store_ds(tmem + T_S, rv, ds);   // over S, read into registers above
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (leader && ok) {
#pragma unroll
      for (int s = 0; s < 8; ++s) {   // dQ += dS K, dS from tensor memory
        mma_f16_ts(tmem + T_ACC0, tmem + T_S + 8 * s, smem_desc(sbase + QQ_K + s * 2048, ATOM, 1024, 2),
                   idesc_bf16(BM, HD) | (1u << 16), (jt > 0 || s > 0) ? 1u : 0u);
      }
      tc_commit(bar(QB_MMA2));
    }
    if (ok) ok = mbar_wait(bar(QB_MMA2), par, ctl, W_MMA2);
    ok = cta_all(ok);
    tc_fence_after();
  }
  if (ok) store_acc(tmem + T_ACC0, a.dq, a, a.Hq, b, hq, it, a.scale);
  if (leader) {
    tc_commit(bar(QB_DRAIN));
    mbar_wait_drain(bar(QB_DRAIN), 0, a.limit_ns);
    if (!qd_seen) mbar_wait_drain(bar(QB_QD), 0, a.limit_ns);
    for (int s2 = 0; s2 < 2; ++s2)
      if (kv_issued[s2] > kv_seen[s2]) mbar_wait_drain(bar(QB_KV0 + s2), (uint32_t)(kv_issued[s2] - 1) & 1u, a.limit_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdArgs& args, cudaStream_t st) {
  static bool attr_set = false;   // the attribute is per function and per process
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KV_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, QQ_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long T = (args.S + BM - 1) / BM;
  const long long rows = (long long)args.B * args.Hq * args.Sp;
  attn_bwd_stats_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(args);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_dq_kernel<<<(unsigned)((long long)args.B * args.Hq * T), kThreads, QQ_SMEM, st>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_kernel<<<(unsigned)((long long)args.B * args.Hkv * T), kThreads, KV_SMEM, st>>>(args);
  return cudaGetLastError();
}

}  // namespace bsc
