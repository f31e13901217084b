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
// The columnwise copy of one 32-token block for four columns d0 = 4 cq .. d0 + 3, this thread's half of
// it: tokens 16 th .. 16 th + 15 at col + r * pitch (r < 16, the four columns' bf16 values as one
// 64-bit word).  The block amax combines with the other half's thread (lane ^ 1).  Returns the 16
// E4M3 bytes of each column's half in out[c] (tokens in natural order) and writes, from the th = 0
// thread, the four scale bytes to vsc[blk_idx * 128 + d0].  Two passes over the rows (the amax, then
// the bytes) keep no column in registers.
__device__ __forceinline__ void colwise_emit(const uint8_t* col, int pitch, int th, long long blk_idx, int cq,
                                             uint8_t* vsc, int rule, uint4 (&out)[4]) {
  uint32_t m01 = 0, m23 = 0;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const uint2 a = *reinterpret_cast<const uint2*>(col + r * pitch);
    asm("max.u16x2 %0, %0, %1;" : "+r"(m01) : "r"(a.x & 0x7FFF7FFFu));
    asm("max.u16x2 %0, %0, %1;" : "+r"(m23) : "r"(a.y & 0x7FFF7FFFu));
  }
  const uint32_t p01 = __shfl_xor_sync(0xFFFFFFFFu, m01, 1), p23 = __shfl_xor_sync(0xFFFFFFFFu, m23, 1);
  asm("max.u16x2 %0, %0, %1;" : "+r"(m01) : "r"(p01));
  asm("max.u16x2 %0, %0, %1;" : "+r"(m23) : "r"(p23));
  float inv0, inv1, inv2, inv3;
  const uint32_t sb0 = e8m0_from_amax(__uint_as_float((m01 & 0xFFFFu) << 16), inv0, rule);
  const uint32_t sb1 = e8m0_from_amax(__uint_as_float(m01 & 0xFFFF0000u), inv1, rule);
  const uint32_t sb2 = e8m0_from_amax(__uint_as_float((m23 & 0xFFFFu) << 16), inv2, rule);
  const uint32_t sb3 = e8m0_from_amax(__uint_as_float(m23 & 0xFFFF0000u), inv3, rule);
  const float2 inv01 = make_float2(inv0, inv1), inv23 = make_float2(inv2, inv3);
  // word i of a column's 16 tokens holds tokens 4i..4i+3 (natural order)
  uint32_t o0[4], o1[4], o2[4], o3[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t01[4], t23[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint2 a = *reinterpret_cast<const uint2*>(col + (4 * i + u) * pitch);
      t01[u] = scale_bf16x2(a.x, inv01);
      t23[u] = scale_bf16x2(a.y, inv23);
    }
    o0[i] = sb0 == 0xFFu ? 0x7F7F7F7Fu
                         : ((uint32_t)cvt_e4m3x2(t01[0].x, t01[1].x) | ((uint32_t)cvt_e4m3x2(t01[2].x, t01[3].x) << 16));
    o1[i] = sb1 == 0xFFu ? 0x7F7F7F7Fu
                         : ((uint32_t)cvt_e4m3x2(t01[0].y, t01[1].y) | ((uint32_t)cvt_e4m3x2(t01[2].y, t01[3].y) << 16));
    o2[i] = sb2 == 0xFFu ? 0x7F7F7F7Fu
                         : ((uint32_t)cvt_e4m3x2(t23[0].x, t23[1].x) | ((uint32_t)cvt_e4m3x2(t23[2].x, t23[3].x) << 16));
    o3[i] = sb3 == 0xFFu ? 0x7F7F7F7Fu
                         : ((uint32_t)cvt_e4m3x2(t23[0].y, t23[1].y) | ((uint32_t)cvt_e4m3x2(t23[2].y, t23[3].y) << 16));
  }
  // the column bytes go through shared memory (the caller's transposed tile), then out in whole rows
  out[0] = make_uint4(o0[0], o0[1], o0[2], o0[3]);
  out[1] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
  out[2] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
  out[3] = make_uint4(o3[0], o3[1], o3[2], o3[3]);
  if (th == 0) *reinterpret_cast<uint32_t*>(vsc + blk_idx * 128 + 4 * cq) = sb0 | (sb1 << 8) | (sb2 << 16) | (sb3 << 24);
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
//     per (b, h, 32-token block, d): vsc[((b*H + h)*(S/32) + s/32)*D + d]; its bytes are
//     transposed in shared memory (over the bf16 tile, once that is read) and written as whole
//     rows of the tile's tokens;
//   * the token-normalised copy in V's own layout with scales vtn_sc[(b*H + h)*S + s].
constexpr int VQ_ROWS = 128;
constexpr int VQ_PITCH = 256 + 16;   // bytes per staged token row
constexpr int VT_PITCH = 128 + 16;   // bytes per d row of the transposed E4M3 tile (in the same buffer)
static_assert(128 * VT_PITCH <= VQ_ROWS * VQ_PITCH, "transposed tile fits");

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

  // load: the whole tile into shared memory by asynchronous 16-byte copies (no registers held while
  // they are in flight), 16 threads per token row; rows past S are filled with zeros
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int c = it * 256 + tid;
    const int r = c >> 4, l16 = c & 15;
    const bool valid = s0 + r < S;
    const long long e = base0 + (long long)(valid ? s0 + r : s0) * row_stride + l16 * 8;
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&tile[r * VQ_PITCH + l16 * 16]);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(v + e * 2), "r"(valid ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  // token-normalised copy from the tile: 8 threads per token row (16 elements each), 32 rows per pass
  if (vtn != nullptr) {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int c = it * 256 + tid;
      const int r = c >> 3, l8 = c & 7;
      if (s0 + r < S) {   // a warp's 4 rows are all valid or all not (S and s0 are multiples of 32)
        const uint4* src = reinterpret_cast<const uint4*>(&tile[r * VQ_PITCH + l8 * 32]);
        const long long e = base0 + (long long)(s0 + r) * row_stride + l8 * 16;
        token_norm_emit(src[0], src[1], e, (long long)plane * S + s0 + r, vtn, vtn_sc, rule, l8);
      }
    }
  }
  if (vt == nullptr) return;

  // columnwise: warp -> (half of the d columns, 32-token block); lane -> (4 columns, half a block)
  const int w = tid >> 5, ln = tid & 31;
  const int th = ln & 1;                    // tokens 16 th .. 16 th + 15 of the block
  const int cq = (w & 1) * 16 + (ln >> 1);  // d = 4 cq .. 4 cq + 3
  const int kb = w >> 1;                    // 32-token block inside the tile (uniform per warp)
  const bool blk_ok = s0 + kb * 32 < S;     // whole 32-token blocks
  uint4 out[4];
  if (blk_ok)
    colwise_emit(&tile[(kb * 32 + 16 * th) * VQ_PITCH + cq * 8], VQ_PITCH, th, (long long)plane * (S / 32) + s0 / 32 + kb,
                 cq, vsc, rule, out);
  __syncthreads();   // every bf16 row is read: the tile now takes the E4M3 bytes as [d][token]
  if (blk_ok) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(&tile[(4 * cq + c) * VT_PITCH + kb * 32 + 16 * th]) = out[c];
  }
  __syncthreads();
  // whole rows of vt: 8 threads per d row (16 bytes each), 32 rows per pass; only the tile's tokens
  const int ntok = min(VQ_ROWS, S - s0);
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int d = it * 32 + (tid >> 3), seg = tid & 7;
    if (seg * 16 < ntok)
      __stcs(reinterpret_cast<uint4*>(vt + ((long long)plane * 128 + d) * S + s0 + seg * 16),
             *reinterpret_cast<const uint4*>(&tile[d * VT_PITCH + seg * 16]));
  }
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
