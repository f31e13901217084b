// MXFP8 quantisers for the attention operands (HBM-bound streaming kernels).
//
// "[PyTorch] Add causal MXFP8 attention without future-token leakage through V scales"
// (TransformerEngine PR #3865), Description:
//   * Q and K are quantised rowwise: E4M3 bytes with one E8M0 scale per 32 elements along D;
//   * V is quantised columnwise: one shared scale per 32 consecutive tokens;
//   * the token-normalised copy of V carries one power-of-two amplitude per token.
// Scale rule (OCP MX, E4M3 elements): scale byte = floor(log2 amax) - 8 + 127, clamped to [0, 254];
// elements x * 2^-e rounded to nearest even on the E4M3 grid, saturating at 448; a block holding a
// NaN or an infinity gets scale 0xFF and element bytes 0x7F.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "bsc_internal.h"

namespace bsc {

// |x| as bf16 bit patterns for 8 packed values; the unsigned maximum of these patterns orders
// finite magnitudes correctly and puts Inf/NaN above every finite value.
__device__ __forceinline__ uint32_t absmax_bits8(const uint4& v) {
  uint32_t a = v.x & 0x7FFF7FFFu, b = v.y & 0x7FFF7FFFu, c = v.z & 0x7FFF7FFFu, d = v.w & 0x7FFF7FFFu;
  uint32_t m;
  asm("max.u16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
  asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(c));
  asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(d));
  return max(m & 0xFFFFu, m >> 16);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two bf16 values of one word times a power of two (exact), as an fp32 pair (low half first).
__device__ __forceinline__ float2 scale_bf16x2(uint32_t w, float2 inv2) {
  return __fmul2_rn(make_float2(bf16_lo(w), bf16_hi(w)), inv2);
}

// 8 bf16 values (one uint4) * inv_scale -> 8 E4M3 bytes (one uint2).
__device__ __forceinline__ uint2 quant8(const uint4& v, float inv, bool nonfinite) {
  if (nonfinite) return make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const float2 inv2 = make_float2(inv, inv);
  uint32_t out[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 a = scale_bf16x2(w[2 * i], inv2), b = scale_bf16x2(w[2 * i + 1], inv2);
    out[i] = (uint32_t)cvt_e4m3x2(a.x, a.y) | ((uint32_t)cvt_e4m3x2(b.x, b.y) << 16);
  }
  return make_uint2(out[0], out[1]);
}

// ------------------------------------------------------------------------------------------
// Rowwise quantiser (Q, K): a CTA of 256 threads takes 64 consecutive tokens s0..s0+63 of one
// (b, h) plane; a token row is 256 bytes = 8 threads x 32 bytes (16 elements) and a 32-element
// block is 2 adjacent threads.  Each thread loads both of its rows (s0 + 32i + tid/8) before
// converting any, so that 64 bytes per thread are in flight.  Scales are compact: the four scale
// bytes of token s (blocks c = d/32) form one 32-bit word at sc[((b*H + h)*S + s)*4 + c].
#define BSC_QUANT_MINB 5   // resident CTAs per SM the register budget is sized for
constexpr int RW_PASSES = 2;                 // token rows per thread
constexpr int RW_ROWS = 32 * RW_PASSES;      // token rows per CTA

// One token row's 16 elements held by this thread (8 threads per row, a 32-element block is 2
// adjacent threads): block amax, scale, E4M3 bytes to q[e..], and the row's scale word from its
// first thread.  Every thread of the warp takes part (the shuffles).
__device__ __forceinline__ void rowwise_emit(const uint4& v0, const uint4& v1, int s, int S, long long e,
                                             long long plane, uint8_t* __restrict__ q, uint8_t* __restrict__ sc,
                                             int rule, int lane, int l8) {
  uint32_t am = max(absmax_bits8(v0), absmax_bits8(v1));
  am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
  float inv;
  const uint32_t sb = e8m0_from_amax(__uint_as_float(am << 16), inv, rule);
  if (s < S) {
    const bool nonfinite = sb == 0xFFu;
    const uint2 lo = quant8(v0, inv, nonfinite), hi = quant8(v1, inv, nonfinite);
    __stcs(reinterpret_cast<uint4*>(q + e), make_uint4(lo.x, lo.y, hi.x, hi.y));
  }
  // gather the 4 block scales of this row on its first thread
  const int base = lane & 24;
  const uint32_t s1 = __shfl_sync(0xFFFFFFFFu, sb, base + 2);
  const uint32_t s2 = __shfl_sync(0xFFFFFFFFu, sb, base + 4);
  const uint32_t s3 = __shfl_sync(0xFFFFFFFFu, sb, base + 6);
  if (s < S && l8 == 0) {
    *reinterpret_cast<uint32_t*>(sc + (plane * S + s) * 4) = sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
  }
}
// The token-normalised copy of one V row (8 threads, 16 elements each; the row valid): one scale
// for the whole row, vtn_sc[row_sc].  Every thread of the 8 takes part (the shuffles).
__device__ __forceinline__ void token_norm_emit(const uint4& v0, const uint4& v1, long long e, long long row_sc,
                                                uint8_t* vtn, uint8_t* vtn_sc, int rule, int l8) {
  uint32_t am = max(absmax_bits8(v0), absmax_bits8(v1));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
  float inv;
  const uint32_t sb = e8m0_from_amax(__uint_as_float(am << 16), inv, rule);
  const bool nonfinite = sb == 0xFFu;
  const uint2 lo = quant8(v0, inv, nonfinite), hi = quant8(v1, inv, nonfinite);
  __stcs(reinterpret_cast<uint4*>(vtn + e), make_uint4(lo.x, lo.y, hi.x, hi.y));
  if (l8 == 0) vtn_sc[row_sc] = (uint8_t)sb;
}
// The columnwise copy of one 32-token block for two columns d0 = 2 dp, d0 + 1: the block's bf16
// values at col + r * pitch (r < 32, the pair as one 32-bit word); writes the 32 bytes of each
// column to vt (transposed: row (plane * 128 + d) of S bytes, tokens s_blk..) and the two scale
// bytes to vsc[blk_idx * 128 + d0].  Two passes over the block (the amax, then the bytes) keep no
// column in registers.
__device__ __forceinline__ void colwise_emit(const uint8_t* col, int pitch, long long plane, int dp, int s_blk,
                                             long long blk_idx, int S, uint8_t* vt, uint8_t* vsc, int rule) {
  uint32_t m = 0;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const uint32_t a = *reinterpret_cast<const uint32_t*>(col + r * pitch) & 0x7FFF7FFFu;
    asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(a));
  }
  float inv0, inv1;
  const uint32_t sb0 = e8m0_from_amax(__uint_as_float((m & 0xFFFFu) << 16), inv0, rule);
  const uint32_t sb1 = e8m0_from_amax(__uint_as_float(m & 0xFFFF0000u), inv1, rule);
  const float2 inv2 = make_float2(inv0, inv1);   // column d0 in the low halves, d1 in the high
  // word i of a column's 32-token block holds tokens 4i..4i+3 (natural order)
  uint32_t o0[8], o1[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float2 t[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) t[u] = scale_bf16x2(*reinterpret_cast<const uint32_t*>(col + (4 * i + u) * pitch), inv2);
    const uint32_t lo0 = cvt_e4m3x2(t[0].x, t[1].x), hi0 = cvt_e4m3x2(t[2].x, t[3].x);
    const uint32_t lo1 = cvt_e4m3x2(t[0].y, t[1].y), hi1 = cvt_e4m3x2(t[2].y, t[3].y);
    o0[i] = sb0 == 0xFFu ? 0x7F7F7F7Fu : (lo0 | (hi0 << 16));
    o1[i] = sb1 == 0xFFu ? 0x7F7F7F7Fu : (lo1 | (hi1 << 16));
  }
  const int d0 = 2 * dp, d1 = 2 * dp + 1;
  uint8_t* row0 = vt + (plane * 128 + d0) * S + s_blk;
  uint8_t* row1 = vt + (plane * 128 + d1) * S + s_blk;
  __stcs(reinterpret_cast<uint4*>(row0), make_uint4(o0[0], o0[1], o0[2], o0[3]));
  __stcs(reinterpret_cast<uint4*>(row0) + 1, make_uint4(o0[4], o0[5], o0[6], o0[7]));
  __stcs(reinterpret_cast<uint4*>(row1), make_uint4(o1[0], o1[1], o1[2], o1[3]));
  __stcs(reinterpret_cast<uint4*>(row1) + 1, make_uint4(o1[4], o1[5], o1[6], o1[7]));
  *reinterpret_cast<uint16_t*>(vsc + blk_idx * 128 + d0) = (uint16_t)(sb0 | (sb1 << 8));
}

// `blk` = plane * ceil(S/64) + s-chunk.
__device__ __forceinline__ void rowwise_rows(const uint8_t* __restrict__ x, uint8_t* __restrict__ q,
                                             uint8_t* __restrict__ sc, int B, int S, int H, int layout, int rule,
                                             long long blk) {
  const int nchunk = (S + RW_ROWS - 1) / RW_ROWS;
  const long long plane = blk / nchunk;
  const int s0 = (int)(blk - plane * nchunk) * RW_ROWS;
  const long long h = plane % H, b = plane / H;
  const long long row_stride = layout == 0 ? (long long)H * 128 : (long long)B * H * 128;   // elements per s
  const long long base0 = layout == 0 ? ((b * S) * H + h) * 128 : (b * H + h) * 128;
  const int tid = threadIdx.x, l8 = tid & 7, lane = tid & 31;
  uint4 v[2 * RW_PASSES];
  long long e[RW_PASSES];
#pragma unroll
  for (int i = 0; i < RW_PASSES; ++i) {
    const int s = s0 + 32 * i + (tid >> 3);
    e[i] = base0 + (long long)s * row_stride + l8 * 16;
    const uint4* src = reinterpret_cast<const uint4*>(x + e[i] * 2);
    v[2 * i] = s < S ? __ldcs(src) : make_uint4(0, 0, 0, 0);
    v[2 * i + 1] = s < S ? __ldcs(src + 1) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < RW_PASSES; ++i)
    rowwise_emit(v[2 * i], v[2 * i + 1], s0 + 32 * i + (tid >> 3), S, e[i], plane, q, sc, rule, lane, l8);
}

__global__ void __launch_bounds__(256, BSC_QUANT_MINB) quant_rowwise_kernel(const uint8_t* __restrict__ x, uint8_t* __restrict__ q,
                                                            uint8_t* __restrict__ sc, int B, int S, int H,
                                                            int layout, int rule) {
  rowwise_rows(x, q, sc, B, S, H, layout, rule, blockIdx.x);
}

// ------------------------------------------------------------------------------------------
// V quantiser: one CTA per (b, h, 128-token tile), 256 threads (the last tile of a sequence may
// hold fewer than 128 tokens, always whole 32-token blocks).  Produces either or both of
//   * the columnwise copy, transposed: vt[((b*H + h)*D + d)*S + s], with compact scales, one byte
//     per (b, h, 32-token block, d): vsc[((b*H + h)*(S/32) + s/32)*D + d];
//   * the token-normalised copy in V's own layout with scales vtn_sc[(b*H + h)*S + s].
constexpr int VQ_ROWS = 128;
constexpr int VQ_PITCH = 256 + 16;   // bytes per staged token row

// `blk` is the (b, h, tile) index; `tile` is VQ_ROWS x VQ_PITCH bytes of shared memory.  The
// whole CTA takes part.
__device__ __forceinline__ void v_tile(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt,
                                       uint8_t* __restrict__ vsc, uint8_t* __restrict__ vtn,
                                       uint8_t* __restrict__ vtn_sc, int B, int S, int H, int layout, int rule,
                                       int blk, uint8_t* tile) {
  const int ntiles = (S + VQ_ROWS - 1) / VQ_ROWS;
  const int tile_idx = blk % ntiles;
  const int plane = blk / ntiles;   // b*H + h
  const int h = plane % H, b = plane / H;
  const int s0 = tile_idx * VQ_ROWS;
  const int tid = threadIdx.x;
  const long long row_stride = layout == 0 ? (long long)H * 128 : (long long)B * H * 128;   // elements per s
  const long long base0 = layout == 0 ? (((long long)b * S) * H + h) * 128 : ((long long)b * H + h) * 128;

  // load: 8 threads per token row (32 bytes each), 32 rows per pass of 256 threads; a warp's 4 rows
  // are all valid or all not (S and s0 are multiples of 32)
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int c = it * 256 + tid;
    const int r = c >> 3, l8 = c & 7;
    const bool valid = s0 + r < S;
    const long long e = base0 + (long long)(s0 + r) * row_stride + l8 * 16;
    const uint4* src = reinterpret_cast<const uint4*>(v + e * 2);
    const uint4 v0 = valid ? __ldcs(src) : make_uint4(0, 0, 0, 0);
    const uint4 v1 = valid ? __ldcs(src + 1) : make_uint4(0, 0, 0, 0);
    uint4* dst = reinterpret_cast<uint4*>(&tile[r * VQ_PITCH + l8 * 32]);
    dst[0] = v0;
    dst[1] = v1;
    // token-normalised copy straight from registers: the 8 threads of a row reduce its amax
    if (vtn != nullptr && valid) token_norm_emit(v0, v1, e, (long long)plane * S + s0 + r, vtn, vtn_sc, rule, l8);
  }
  if (vt == nullptr) return;
  __syncthreads();

  // columnwise: thread -> (pair of d columns, 32-token block)
  const int dp = tid & 63;      // d = 2*dp, 2*dp + 1
  const int kb = tid >> 6;      // 32-token block inside the tile
  if (s0 + kb * 32 < S)   // whole 32-token blocks
    colwise_emit(&tile[kb * 32 * VQ_PITCH + dp * 4], VQ_PITCH, plane, dp, s0 + kb * 32,
                 (long long)plane * (S / 32) + s0 / 32 + kb, S, vt, vsc, rule);
}

__global__ void __launch_bounds__(256, BSC_QUANT_MINB) quant_v_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt,
                                                      uint8_t* __restrict__ vsc, uint8_t* __restrict__ vtn,
                                                      uint8_t* __restrict__ vtn_sc, int B, int S, int H,
                                                      int layout, int rule) {
  __shared__ __align__(16) uint8_t tile[VQ_ROWS * VQ_PITCH];
  v_tile(v, vt, vsc, vtn, vtn_sc, B, S, H, layout, rule, (int)blockIdx.x, tile);
}

// ------------------------------------------------------------------------------------------
// Q, K and V in one launch: CTAs [0, nv) take V tiles, then Q's 64-token chunks, then K's.  Each
// CTA does exactly what the matching kernel above does for the same index.
__global__ void __launch_bounds__(256, BSC_QUANT_MINB) quant_qkv_kernel(const __grid_constant__ QkvQuantArgs a) {
  __shared__ __align__(16) uint8_t tile[VQ_ROWS * VQ_PITCH];
  const long long blk = blockIdx.x;
  if (blk < a.nv_blocks) {
    v_tile(reinterpret_cast<const uint8_t*>(a.v), a.vt, a.vsc, a.vtn, a.vtn_sc, a.B, a.S, a.Hkv, a.layout, a.rule,
           (int)blk, tile);
  } else if (blk < a.nv_blocks + a.nq_blocks) {
    rowwise_rows(reinterpret_cast<const uint8_t*>(a.q), a.q8, a.q_sc, a.B, a.S, a.Hq, a.layout, a.rule,
                 blk - a.nv_blocks);
  } else {
    rowwise_rows(reinterpret_cast<const uint8_t*>(a.k), a.k8, a.k_sc, a.B, a.S, a.Hkv, a.layout, a.rule,
                 blk - a.nv_blocks - a.nq_blocks);
  }
}

// ------------------------------------------------------------------------------------------
cudaError_t launch_quant_rowwise(const void* x, uint8_t* q, uint8_t* sc, int B, int S, int H, int layout,
                                 cudaStream_t st, int rule) {
  const long long grid = (long long)B * H * ((S + RW_ROWS - 1) / RW_ROWS);
  quant_rowwise_kernel<<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const uint8_t*>(x), q, sc, B, S, H, layout,
                                                        rule);
  return cudaGetLastError();
}

cudaError_t launch_quant_qkv(QkvQuantArgs a, cudaStream_t st) {
  const long long nchunk = (a.S + RW_ROWS - 1) / RW_ROWS;
  a.nv_blocks = (long long)a.B * a.Hkv * ((a.S + VQ_ROWS - 1) / VQ_ROWS);
  a.nq_blocks = (long long)a.B * a.Hq * nchunk;
  const long long nk_blocks = (long long)a.B * a.Hkv * nchunk;
  quant_qkv_kernel<<<(unsigned)(a.nv_blocks + a.nq_blocks + nk_blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quant_v(const void* v, uint8_t* vt, uint8_t* vsc, uint8_t* vtn, uint8_t* vtn_sc, int B, int S,
                           int H, int layout, cudaStream_t st, int rule) {
  const long long ctas = (long long)B * H * ((S + VQ_ROWS - 1) / VQ_ROWS);
  quant_v_kernel<<<(unsigned)ctas, 256, 0, st>>>(reinterpret_cast<const uint8_t*>(v), vt, vsc, vtn, vtn_sc, B, S,
                                                  H, layout, rule);
  return cudaGetLastError();
}

}  // namespace bsc
