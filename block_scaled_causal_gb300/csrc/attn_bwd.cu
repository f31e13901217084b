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

enum Site : int { W_KV = 0x20, W_QD, W_MMA1, W_MMA2, W_MMA3, W_DO };

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

// Row statistics of the 128 query rows of tile `it`: LSE in log2 units and Dlt = <dO_i, O_i>.
// Two threads per row, 64 head-dim elements each.  Rows past S get LSE = +inf and Dlt = 0, which
// makes their P and dS exactly 0.
__device__ __forceinline__ void row_stats(const BwdArgs& a, int b, int hq, int it, float* lse2, float* dlt) {
  const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int i = it * BM + r;
  float acc = 0.f;
  if (i < a.S) {
    const long long row = a.layout == 0 ? ((long long)b * a.S + i) * a.Hq + hq : ((long long)i * a.B + b) * a.Hq + hq;
    const uint4* po = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.o) + row * HD + 64 * half);
    const uint4* pd = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.dO) + row * HD + 64 * half);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 x = __ldg(po + c), y = __ldg(pd + c);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), acc);
        acc = fmaf(__uint_as_float(xs[e] & 0xFFFF0000u), __uint_as_float(ys[e] & 0xFFFF0000u), acc);
      }
    }
  }
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
  if (half == 0) {
    dlt[r] = i < a.S ? acc : 0.f;
    lse2[r] = i < a.S ? a.lse[((long long)b * a.Hq + hq) * a.S + i] * 1.4426950408889634f : INFINITY;
  }
}

// The same statistics from shared memory: the BF16 tiles of dO and O (TMA zero-fills rows past
// S) and the tile's LSE values (copied for the rows below S only).
__device__ __forceinline__ void row_stats_tiles(const BwdArgs& a, int it, const uint8_t* do_tile,
                                                const uint8_t* o_tile, const float* lse_tile, float* lse2,
                                                float* dlt) {
  const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int i = it * BM + r;
  float acc = 0.f;
  if (i < a.S) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t off = bf_off((uint32_t)r, (uint32_t)(64 * half + 8 * c));
      const uint4 x = *reinterpret_cast<const uint4*>(o_tile + off);
      const uint4 y = *reinterpret_cast<const uint4*>(do_tile + off);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), acc);
        acc = fmaf(__uint_as_float(xs[e] & 0xFFFF0000u), __uint_as_float(ys[e] & 0xFFFF0000u), acc);
      }
    }
  }
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
  if (half == 0) {
    dlt[r] = i < a.S ? acc : 0.f;
    lse2[r] = i < a.S ? lse_tile[r] * 1.4426950408889634f : INFINITY;
  }
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
// S = Qh Kh^T from E4M3 tiles and row-atom scales (copied to TMEM columns t_sf.. first).
__device__ __forceinline__ void mma_s(uint32_t tmem, uint32_t t_sf, uint32_t q8, uint32_t k8, uint32_t sfq,
                                      uint32_t sfk) {
  tc_cp_32x128b_warpx4(tmem + t_sf, desc_sf_block(sfq));
  tc_cp_32x128b_warpx4(tmem + t_sf + 4, desc_sf_block(sfk));
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    mma_mxf8_ss(tmem + T_S, desc_kmajor_sw128(q8 + kk * 32), desc_kmajor_sw128(k8 + kk * 32),
                idesc_mxf8(BM, BN, kk, kk), tmem + t_sf, tmem + t_sf + 4, kk > 0 ? 1u : 0u);
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
// A thread's 64 values as BF16 into a [q][key] tile: keys 8k + 2qd and 8k + 2qd + 1 are adjacent,
// one 32-bit store per pair.
__device__ __forceinline__ void store_rows(uint8_t* tile, const RowView& rv, const float (&x)[64]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int key = 8 * k + 2 * rv.qd;
    *reinterpret_cast<uint32_t*>(tile + bf_off(rv.ra, key)) = pack_bf16x2(x[4 * k], x[4 * k + 1]);
    *reinterpret_cast<uint32_t*>(tile + bf_off(rv.rb, key)) = pack_bf16x2(x[4 * k + 2], x[4 * k + 3]);
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
// dK, dV.  Shared memory (bytes from a 1024-aligned base):
constexpr uint32_t KV_K8 = 0;                 // K bytes [key][d], swizzled
constexpr uint32_t KV_V = KV_K8 + 16384;      // V bf16 [key][d]
constexpr uint32_t KV_Q8 = KV_V + 32768;      // Q bytes [q][d], swizzled
constexpr uint32_t KV_Q = KV_Q8 + 16384;      // Q bf16 [q][d]
constexpr uint32_t KV_DO = KV_Q + 32768;      // dO bf16 [q][d]
constexpr uint32_t KV_P = KV_DO + 32768;      // P bf16 [q][key] (the V bytes [key][d] before that)
constexpr uint32_t KV_VN8 = KV_P;
constexpr uint32_t KV_DS = KV_P + 32768;      // dS bf16 [q][key] (O bf16 [q][d] before that)
constexpr uint32_t KV_SFQ = KV_DS + 32768;     // compact Q scales of the tile
constexpr uint32_t KV_SFK = KV_SFQ + 512;      // compact K scales
constexpr uint32_t KV_SFQA = KV_SFK + 512;     // the same as scale-factor atoms
constexpr uint32_t KV_SFKA = KV_SFQA + 512;
constexpr uint32_t KV_AMP = KV_SFKA + 512;
constexpr uint32_t KV_STAT = KV_AMP + 128;    // [2 buffers][LSE | Dlt][128] floats
constexpr uint32_t KV_LSE = KV_STAT + 2048;
constexpr uint32_t KV_BAR = KV_LSE + 512;
constexpr uint32_t KV_MISC = KV_BAR + 64;
constexpr uint32_t KV_SMEM = KV_MISC + 16 + 1024;
static_assert(KV_SMEM <= 227 * 1024, "shared memory budget");
enum KvBar : uint32_t { KB_KV = 0, KB_Q, KB_DO, KB_MMA1, KB_MMA2, KB_MMA3, KB_DRAIN, KB_COUNT };

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](uint32_t i) { return sbase + KV_BAR + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + KV_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + KV_MISC + 4);
  auto stat = [&](int buf) { return reinterpret_cast<float*>(smem + KV_STAT) + buf * 256; };

  const int T = (a.S + BN - 1) / BN;
  const int g = a.Hq / a.Hkv;
  // key tiles with the most query tiles first
  const int bh = blockIdx.x % (a.B * a.Hkv);
  const int jt = (int)(blockIdx.x / (a.B * a.Hkv));
  const int hk = bh % a.Hkv, b = bh / a.Hkv;
  const long long kv_plane = (long long)b * a.Hkv + hk;
  const int nkeys = min(BN, a.S - jt * BN);
  const int n_iter = g * (T - jt);   // (query head, query tile) pairs

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < KB_COUNT; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(sbase + KV_MISC, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, a.dev_status, a.limit_ns};
  const bool leader = threadIdx.x == 0;
  // Query tiles from the last down to the key tile, the group's heads innermost: CTAs of one KV head
  // that run at the same time then read the same Q, dO and O tiles, which stay in L2.
  auto hq_of = [&](int n) { return hk * g + n % g; };
  auto it_of = [&](int n) { return T - 1 - n / g; };
  auto load_q = [&](int n) {
    const uint32_t nr = (uint32_t)min(BM, a.S - it_of(n) * BM);
    mbar_arrive_expect_tx(bar(KB_Q), BM * HD + 4 * nr);
    tma_load_4d(sbase + KV_Q8, &a.tm_q, bar(KB_Q), 0, hq_of(n), it_of(n) * BM, b);
    bulk_load(sbase + KV_SFQ, a.q_sc + (((long long)b * a.Hq + hq_of(n)) * a.S + (long long)it_of(n) * BM) * 4, 4 * nr,
              bar(KB_Q));
  };
  // dO into its tile and O into the dS tile (read for the row statistics before dS is written)
  auto load_do = [&](int n) {
    const int it = it_of(n);
    const uint32_t lse_bytes = 4u * (uint32_t)min(BM, a.S - it * BM);
    mbar_arrive_expect_tx(bar(KB_DO), 4 * BM * HD + lse_bytes);
    tma_load_4d(sbase + KV_DO, &a.tm_do, bar(KB_DO), 0, hq_of(n), it * BM, b);
    tma_load_4d(sbase + KV_DO + ATOM, &a.tm_do, bar(KB_DO), 64, hq_of(n), it * BM, b);
    tma_load_4d(sbase + KV_DS, &a.tm_o, bar(KB_DO), 0, hq_of(n), it * BM, b);
    tma_load_4d(sbase + KV_DS + ATOM, &a.tm_o, bar(KB_DO), 64, hq_of(n), it * BM, b);
    bulk_load(sbase + KV_LSE, a.lse + ((long long)b * a.Hq + hq_of(n)) * a.S + (long long)it * BM, lse_bytes,
              bar(KB_DO));
  };
  bool ok = true;
  int q_issued = 0, q_seen = 0, do_issued = 0, do_seen = 0;

  // this CTA's K and V tiles, and the first query tile
  if (leader) {
    mbar_arrive_expect_tx(bar(KB_KV), 2 * BN * HD + 4 * (uint32_t)nkeys + (uint32_t)nkeys);
    tma_load_4d(sbase + KV_K8, &a.tm_k, bar(KB_KV), 0, hk, jt * BN, b);
    bulk_load(sbase + KV_SFK, a.k_sc + (kv_plane * a.S + (long long)jt * BN) * 4, 4 * (uint32_t)nkeys, bar(KB_KV));
    tma_load_4d(sbase + KV_VN8, &a.tm_vtn, bar(KB_KV), 0, hk, jt * BN, b);
    bulk_load(sbase + KV_AMP, a.vtn_sc + kv_plane * a.S + (long long)jt * BN, (uint32_t)nkeys, bar(KB_KV));
    load_q(0);
    load_do(0);
  }
  q_issued = do_issued = 1;
  ok = cta_all(mbar_wait(bar(KB_KV), 0, ctl, W_KV));
  const bool kv_seen = ok;
  if (ok) {
    if (threadIdx.x < 32) rows_to_atom(smem + KV_SFK, smem + KV_SFKA, nkeys, threadIdx.x);
    decode_vt(smem + KV_VN8, smem + KV_AMP, smem + KV_V, nkeys);
  }
  __syncthreads();   // the V bytes are read before P overwrites them

  const RowView rv = row_view();
  for (int n = 0; n < n_iter; ++n) {
    const uint32_t par = (uint32_t)n & 1u;
    const int it = it_of(n);
    float* lse2 = stat(n & 1);
    float* dlt = lse2 + 128;
    if (ok) ok = mbar_wait(bar(KB_Q), par, ctl, W_QD);
    ok = cta_all(ok);
    if (ok) ++q_seen;
    if (ok && threadIdx.x < 32) rows_to_atom(smem + KV_SFQ, smem + KV_SFQA, min(BM, a.S - it * BM), threadIdx.x);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // S first (it reads the E4M3 bytes); its scale factors occupy dP's first columns until it has
    // completed
    if (leader && ok) {
      mma_s(tmem, T_DP, sbase + KV_Q8, sbase + KV_K8, sbase + KV_SFQA, sbase + KV_SFKA);
      tc_commit(bar(KB_MMA1));
    }
    // Q decoded to BF16 for the dK MMA while S computes (the previous dK MMA, the last reader of the
    // BF16 tile, completed before this iteration)
    if (ok) decode_rows(smem + KV_Q8, smem + KV_SFQ, smem + KV_Q, min(BM, a.S - it * BM));
    if (ok) ok = mbar_wait(bar(KB_MMA1), par, ctl, W_MMA1);
    ok = cta_all(ok);
    tc_fence_after();
    if (ok) ok = mbar_wait(bar(KB_DO), par, ctl, W_DO);
    ok = cta_all(ok);
    if (ok) ++do_seen;
    if (leader && ok) {
      if (n + 1 < n_iter) {   // the Q bytes are free again: fetch the next query tile's
        load_q(n + 1);
        ++q_issued;
      }
      mma_bf16_k128<false, false>(tmem + T_DP, sbase + KV_DO, sbase + KV_V, false);   // dP = dO V^T
      tc_commit(bar(KB_MMA3));
    }
    // LSE and Dlt of this query tile while dP computes (dO and O are in shared memory by now)
    if (ok) row_stats_tiles(a, it, smem + KV_DO, smem + KV_DS, reinterpret_cast<const float*>(smem + KV_LSE), lse2, dlt);
    __syncthreads();   // O's tile is read before dS overwrites it
    float p[64];
    if (ok) {
      compute_p(tmem, rv, lse2, a.scale_log2e, it == jt, p);
      store_rows(smem + KV_P, rv, p);
    }
    if (ok) ok = mbar_wait(bar(KB_MMA3), par, ctl, W_MMA3);
    ok = cta_all(ok);
    tc_fence_after();
    if (ok) {
      float ds[64];
      compute_ds(tmem, rv, dlt, p, ds);
      store_rows(smem + KV_DS, rv, ds);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (leader && ok) {
      mma_bf16_k128<true, true>(tmem + T_ACC0, sbase + KV_P, sbase + KV_DO, n > 0);   // dV += P^T dO
      mma_bf16_k128<true, true>(tmem + T_ACC1, sbase + KV_DS, sbase + KV_Q, n > 0);   // dK += dS^T Q
      tc_commit(bar(KB_MMA2));
    }
    if (ok) ok = mbar_wait(bar(KB_MMA2), par, ctl, W_MMA2);
    ok = cta_all(ok);
    tc_fence_after();
    if (leader && ok && n + 1 < n_iter) {   // dO is free again
      load_do(n + 1);
      ++do_issued;
    }
  }
  if (ok && n_iter > 0) {
    store_acc(tmem + T_ACC0, a.dv, a, a.Hkv, b, hk, jt, 1.0f);
    store_acc(tmem + T_ACC1, a.dk, a, a.Hkv, b, hk, jt, a.scale);
  }
  if (leader) {
    // every tcgen05 operation and copy this thread issued must finish before the CTA exits
    tc_commit(bar(KB_DRAIN));
    mbar_wait_drain(bar(KB_DRAIN), 0, a.limit_ns);
    if (!kv_seen) mbar_wait_drain(bar(KB_KV), 0, a.limit_ns);
    if (q_issued > q_seen) mbar_wait_drain(bar(KB_Q), (uint32_t)(q_issued - 1) & 1u, a.limit_ns);
    if (do_issued > do_seen) mbar_wait_drain(bar(KB_DO), (uint32_t)(do_issued - 1) & 1u, a.limit_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(tmem, 512);
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
  row_stats(a, b, hq, it, lse2, dlt);
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
  attn_bwd_dq_kernel<<<(unsigned)((long long)args.B * args.Hq * T), kThreads, QQ_SMEM, st>>>(args);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_kernel<<<(unsigned)((long long)args.B * args.Hkv * T), kThreads, KV_SMEM, st>>>(args);
  return cudaGetLastError();
}

}  // namespace bsc
