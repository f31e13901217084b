// C-ABI entry points: argument checks, tensor-map creation, launches.  See include/bsc.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/bsc.h"
#include "bsc_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device capability check, cached per device ordinal.
bsc_status check_device() {
  static std::mutex mu;
  static int cached[64];   // 0 unknown, 1 ok, 2 bad
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSC_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BSC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return BSC_ERR_CUDA;
    cached[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return cached[dev] == 1 ? BSC_OK : BSC_ERR_UNSUPPORTED;
}

// Common shape checks.  Returns BSC_OK with *empty set when there is nothing to do.
bsc_status check_shape(int B, int S, int H, int D, int layout, bool* empty) {
  *empty = false;
  if (B < 0 || S < 0 || H < 0 || D < 0) return BSC_ERR_SHAPE;
  if (layout != BSC_BSHD && layout != BSC_SBHD) return BSC_ERR_SHAPE;
  if (B == 0 || S == 0 || H == 0) {
    *empty = true;
    return BSC_OK;
  }
  if (D != 128 || S % 32 != 0) return BSC_ERR_UNSUPPORTED;
  // every index the kernels form fits in 64 bits; the grids (one CTA per 64 tokens of a (b, h) plane
  // at most) must fit their limits
  if ((long long)B * H * ((S + 63) / 64) >= (1LL << 31)) return BSC_ERR_UNSUPPORTED;
  return BSC_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// E4M3 [.., S, .., H, 128] operand as a 4-D map {D, H, S, B} with a 128-token x 128-byte box.
bool encode_tokens_map(CUtensorMap* m, const void* base, int B, int S, int H, int layout, bool swizzle) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  const cuuint64_t sH = 128;
  const cuuint64_t sS = layout == BSC_BSHD ? (cuuint64_t)H * 128 : (cuuint64_t)B * H * 128;
  const cuuint64_t sB = layout == BSC_BSHD ? (cuuint64_t)S * H * 128 : (cuuint64_t)H * 128;
  const cuuint64_t strides[3] = {sH, sS, sB};
  const cuuint32_t box[4] = {128, 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 [.., S, .., H, 128] tensor as a 4-D map {D, H, S, B} with a 128-token x 64-element box
// (128 bytes, the swizzle span): two boxes cover a row's 128 elements.
bool encode_bf16_tokens_map(CUtensorMap* m, const void* base, int B, int S, int H, int layout) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  const cuuint64_t sH = 256;
  const cuuint64_t sS = layout == BSC_BSHD ? (cuuint64_t)H * 256 : (cuuint64_t)B * H * 256;
  const cuuint64_t sB = layout == BSC_BSHD ? (cuuint64_t)S * H * 256 : (cuuint64_t)H * 256;
  const cuuint64_t strides[3] = {sH, sS, sB};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 planes [planes][rows][128] (the backward's workspace) as a 3-D map with a 64-element x
// 128-row box and the 128-byte swizzle: two boxes cover a tile's 128 columns.
bool encode_bf16_planar_map(CUtensorMap* m, void* base, long long planes, int rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {256, (cuuint64_t)rows * 256};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Transposed V bytes [rows = B*H*D][S] as a 2-D map with a 128-key x 128-row box.
bool encode_vt_map(CUtensorMap* m, const void* base, long long rows, int S) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)S, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)S};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bsc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BSC_OK : BSC_ERR_CUDA; }

bsc_status quant_v_common(const void* v, int B, int S, int H, int D, bsc_layout layout, uint8_t* vt, uint8_t* vsc,
                          uint8_t* vtn, uint8_t* vtn_sc, bsc_stream_t stream, bool want_col, bool want_tn,
                          int rule = 0) {
  bool empty;
  bsc_status s = check_shape(B, S, H, D, layout, &empty);
  if (s != BSC_OK || empty) return s;
  if (!v || (want_col && (!vt || !vsc)) || (want_tn && (!vtn || !vtn_sc))) return BSC_ERR_NULL;
  if (!aligned16(v) || (want_col && (!aligned16(vt) || !aligned16(vsc))) ||
      (want_tn && (!aligned16(vtn) || !aligned16(vtn_sc))))
    return BSC_ERR_ALIGN;
  if ((s = check_device()) != BSC_OK) return s;
  return from_cuda(bsc::launch_quant_v(v, want_col ? vt : nullptr, want_col ? vsc : nullptr,
                                       want_tn ? vtn : nullptr, want_tn ? vtn_sc : nullptr, B, S, H, layout,
                                       reinterpret_cast<cudaStream_t>(stream), rule));
}

}  // namespace

extern "C" {

int bsc_abi_version(void) { return 3; }

const char* bsc_status_string(bsc_status s) {
  switch (s) {
    case BSC_OK: return "BSC_OK";
    case BSC_ERR_NULL: return "BSC_ERR_NULL: a required pointer is NULL";
    case BSC_ERR_SHAPE: return "BSC_ERR_SHAPE: invalid sizes, head grouping or layout";
    case BSC_ERR_ALIGN: return "BSC_ERR_ALIGN: a pointer is not 16-byte aligned";
    case BSC_ERR_UNSUPPORTED: return "BSC_ERR_UNSUPPORTED: unsupported size, option or device";
    case BSC_ERR_CUDA: return "BSC_ERR_CUDA: a CUDA call failed";
    case BSC_ERR_DEVICE_TIMEOUT: return "BSC_ERR_DEVICE_TIMEOUT: a device-side wait gave up";
  }
  return "unknown bsc_status";
}

bsc_status mxfp8_quantize_qk_rowwise(const void* x, int B, int S, int H, int D, bsc_layout layout, uint8_t* xq,
                                     uint8_t* xsc, bsc_stream_t stream) {
  bool empty;
  bsc_status s = check_shape(B, S, H, D, layout, &empty);
  if (s != BSC_OK || empty) return s;
  if (!x || !xq || !xsc) return BSC_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(xsc)) return BSC_ERR_ALIGN;
  if ((s = check_device()) != BSC_OK) return s;
  return from_cuda(bsc::launch_quant_rowwise(x, xq, xsc, B, S, H, layout, reinterpret_cast<cudaStream_t>(stream)));
}

bsc_status mxfp8_quantize(const bsc_quant_params* p, bsc_stream_t stream) {
  if (!p) return BSC_ERR_NULL;
  if (p->rule != BSC_SCALE_FLOOR && p->rule != BSC_SCALE_CEIL) return BSC_ERR_UNSUPPORTED;
  const bsc_layout layout = (bsc_layout)p->layout;
  switch (p->kind) {
    case BSC_QUANT_ROWWISE: {
      bool empty;
      bsc_status s = check_shape(p->B, p->S, p->H, p->D, p->layout, &empty);
      if (s != BSC_OK || empty) return s;
      if (!p->x || !p->e4m3 || !p->sc) return BSC_ERR_NULL;
      if (!aligned16(p->x) || !aligned16(p->e4m3) || !aligned16(p->sc)) return BSC_ERR_ALIGN;
      if ((s = check_device()) != BSC_OK) return s;
      return from_cuda(bsc::launch_quant_rowwise(p->x, p->e4m3, p->sc, p->B, p->S, p->H, p->layout,
                                                 reinterpret_cast<cudaStream_t>(stream), p->rule));
    }
    case BSC_QUANT_V_COLWISE:
      return quant_v_common(p->x, p->B, p->S, p->H, p->D, layout, p->e4m3, p->sc, nullptr, nullptr, stream, true,
                            false, p->rule);
    case BSC_QUANT_V_TOKEN_NORM:
      return quant_v_common(p->x, p->B, p->S, p->H, p->D, layout, nullptr, nullptr, p->vtn_e4m3, p->vtn_sc, stream,
                            false, true, p->rule);
    case BSC_QUANT_V_FUSED:
      return quant_v_common(p->x, p->B, p->S, p->H, p->D, layout, p->e4m3, p->sc, p->vtn_e4m3, p->vtn_sc, stream,
                            true, true, p->rule);
    default:
      return BSC_ERR_UNSUPPORTED;
  }
}

bsc_status mxfp8_quantize_v_colwise(const void* v, int B, int S, int H, int D, bsc_layout layout, uint8_t* vt,
                                    uint8_t* vsc, bsc_stream_t stream) {
  return quant_v_common(v, B, S, H, D, layout, vt, vsc, nullptr, nullptr, stream, true, false);
}

bsc_status v_token_normalize(const void* v, int B, int S, int H, int D, bsc_layout layout, uint8_t* vtn,
                             uint8_t* vtn_sc, bsc_stream_t stream) {
  return quant_v_common(v, B, S, H, D, layout, nullptr, nullptr, vtn, vtn_sc, stream, false, true);
}

bsc_status mxfp8_quantize_v_fused(const void* v, int B, int S, int H, int D, bsc_layout layout, uint8_t* vt,
                                  uint8_t* vsc, uint8_t* vtn, uint8_t* vtn_sc, bsc_stream_t stream) {
  return quant_v_common(v, B, S, H, D, layout, vt, vsc, vtn, vtn_sc, stream, true, true);
}

bsc_status mxfp8_quantize_qkv(const bsc_qkv_quant_params* p, bsc_stream_t stream) {
  if (!p) return BSC_ERR_NULL;
  if (p->Hq < 0 || p->Hkv < 0) return BSC_ERR_SHAPE;
  if (p->rule != BSC_SCALE_FLOOR && p->rule != BSC_SCALE_CEIL) return BSC_ERR_UNSUPPORTED;
  bool empty;
  bsc_status s = check_shape(p->B, p->S, p->Hq, p->D, p->layout, &empty);
  if (s != BSC_OK) return s;
  if (!empty && p->Hkv == 0) return BSC_ERR_SHAPE;
  if (empty) return BSC_OK;
  if (p->Hq % p->Hkv != 0) return BSC_ERR_SHAPE;
  // one launch: V tiles plus Q's and K's 64-token chunks
  if ((long long)p->B * (p->Hq + 2LL * p->Hkv) * ((p->S + 63) / 64) >= (1LL << 31)) return BSC_ERR_UNSUPPORTED;
  const bool col = p->v_e4m3_t != nullptr || p->v_sc != nullptr;
  const bool tn = p->vtn_e4m3 != nullptr || p->vtn_sc != nullptr;
  if (!p->q || !p->k || !p->v || !p->q_e4m3 || !p->q_sc || !p->k_e4m3 || !p->k_sc) return BSC_ERR_NULL;
  if ((col && (!p->v_e4m3_t || !p->v_sc)) || (tn && (!p->vtn_e4m3 || !p->vtn_sc)) || (!col && !tn))
    return BSC_ERR_NULL;
  for (const void* ptr : {p->q, p->k, p->v, (const void*)p->q_e4m3, (const void*)p->q_sc, (const void*)p->k_e4m3,
                          (const void*)p->k_sc, (const void*)p->v_e4m3_t, (const void*)p->v_sc,
                          (const void*)p->vtn_e4m3, (const void*)p->vtn_sc})
    if (!aligned16(ptr)) return BSC_ERR_ALIGN;
  if ((s = check_device()) != BSC_OK) return s;
  bsc::QkvQuantArgs a{};
  a.q = p->q;
  a.k = p->k;
  a.v = p->v;
  a.B = p->B;
  a.S = p->S;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.layout = p->layout;
  a.rule = p->rule;
  a.q8 = p->q_e4m3;
  a.q_sc = p->q_sc;
  a.k8 = p->k_e4m3;
  a.k_sc = p->k_sc;
  a.vt = p->v_e4m3_t;
  a.vsc = p->v_sc;
  a.vtn = p->vtn_e4m3;
  a.vtn_sc = p->vtn_sc;
  return from_cuda(bsc::launch_quant_qkv(a, reinterpret_cast<cudaStream_t>(stream)));
}

bsc_status mxfp8_causal_attn_fwd(const bsc_attn_fwd_params* p, bsc_stream_t stream) {
  if (!p) return BSC_ERR_NULL;
  if (p->Hq < 0 || p->Hkv < 0) return BSC_ERR_SHAPE;
  bool empty;
  bsc_status s = check_shape(p->B, p->S, p->Hq, p->D, p->layout, &empty);
  if (s != BSC_OK) return s;
  if (!empty && p->Hkv == 0) return BSC_ERR_SHAPE;
  if (empty) return BSC_OK;
  if (p->Hq % p->Hkv != 0) return BSC_ERR_SHAPE;
  if (p->p_terms != 1 && p->p_terms != 2) return BSC_ERR_UNSUPPORTED;
  if (p->leaky != 0 && p->leaky != 1) return BSC_ERR_UNSUPPORTED;
  // the kernel takes row maxima of the raw scores before scaling: a positive, finite scale only
  if (!(std::isfinite(p->softmax_scale) && p->softmax_scale > 0.f)) return BSC_ERR_UNSUPPORTED;
  const bool own = p->leaky == 0;
  if (!p->q || !p->q_sc || !p->k || !p->k_sc || !p->v_t || !p->v_sc || !p->lse) return BSC_ERR_NULL;
  if (!p->o && !p->o_e4m3) return BSC_ERR_NULL;
  if (p->o_e4m3 && !p->o_sc) return BSC_ERR_NULL;
  if (own && (!p->vtn || !p->vtn_sc)) return BSC_ERR_NULL;
  const void* ptrs[] = {p->q, p->q_sc, p->k, p->k_sc, p->v_t, p->v_sc, p->o, p->lse, p->dev_status,
                        p->o_e4m3, p->o_sc};
  for (const void* q : ptrs)
    if (!aligned16(q)) return BSC_ERR_ALIGN;
  if (own && (!aligned16(p->vtn) || !aligned16(p->vtn_sc))) return BSC_ERR_ALIGN;
  if ((s = check_device()) != BSC_OK) return s;

  bsc::AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!encode_tokens_map(&a.tm_q, p->q, p->B, p->S, p->Hq, p->layout, true) ||
      !encode_tokens_map(&a.tm_k, p->k, p->B, p->S, p->Hkv, p->layout, true) ||
      !encode_vt_map(&a.tm_v, p->v_t, (long long)p->B * p->Hkv * 128, p->S))
    return BSC_ERR_CUDA;
  a.q_sc = p->q_sc;
  a.k_sc = p->k_sc;
  a.v_sc = p->v_sc;
  a.vtn = own ? p->vtn : nullptr;
  a.vtn_sc = own ? p->vtn_sc : nullptr;
  a.o = p->o;
  a.o8 = p->o_e4m3;
  a.o_sc = p->o_sc;
  a.lse = p->lse;
  a.dev_status = p->dev_status;
  a.limit_ns = (unsigned long long)(p->wait_timeout_ms ? p->wait_timeout_ms : 2000u) * 1000000ull;
  a.B = p->B;
  a.S = p->S;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.layout = p->layout;
  a.scale_log2e = (float)((double)p->softmax_scale * 1.4426950408889634);
  a.p_terms = p->p_terms;
  a.leaky = p->leaky;
  a.inject_stall = p->debug_stall ? 1 : 0;
  return from_cuda(bsc::launch_attn_fwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t bf16_attn_bwd_workspace_bytes(int B, int S, int Hq, int Hkv) {
  if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0) return 0;
  return bsc::bwd_workspace_bytes(B, S, Hq, Hkv);
}

bsc_status bf16_attn_bwd(const bsc_attn_bwd_params* p, bsc_stream_t stream) {
  if (!p) return BSC_ERR_NULL;
  if (p->Hq < 0 || p->Hkv < 0) return BSC_ERR_SHAPE;
  bool empty;
  bsc_status s = check_shape(p->B, p->S, p->Hq, p->D, p->layout, &empty);
  if (s != BSC_OK) return s;
  if (!empty && p->Hkv == 0) return BSC_ERR_SHAPE;
  if (empty) return BSC_OK;
  if (p->Hq % p->Hkv != 0) return BSC_ERR_SHAPE;
  if (!(std::isfinite(p->softmax_scale) && p->softmax_scale > 0.f)) return BSC_ERR_UNSUPPORTED;
  if (!p->q || !p->q_sc || !p->k || !p->k_sc || !p->vtn || !p->vtn_sc || !p->o || !p->lse || !p->d_o || !p->dq ||
      !p->dk || !p->dv || !p->workspace)
    return BSC_ERR_NULL;
  const void* ptrs[] = {p->q,  p->q_sc, p->k,  p->k_sc, p->vtn,       p->vtn_sc,    p->o,
                        p->lse, p->d_o, p->dq, p->dk,   p->dv, p->workspace, p->dev_status};
  for (const void* q : ptrs)
    if (!aligned16(q)) return BSC_ERR_ALIGN;
  if (p->workspace_bytes < bf16_attn_bwd_workspace_bytes(p->B, p->S, p->Hq, p->Hkv)) return BSC_ERR_SHAPE;
  if ((s = check_device()) != BSC_OK) return s;

  bsc::BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const int Sp = (p->S + 127) / 128 * 128;
  const long long rq = (long long)p->B * p->Hq * Sp, rk = (long long)p->B * p->Hkv * Sp;
  uint8_t* ws = reinterpret_cast<uint8_t*>(p->workspace);
  a.ws = p->workspace;
  a.qh = reinterpret_cast<uint16_t*>(ws + 8 * rq);
  a.kh = a.qh + rq * 128;
  a.vh = a.kh + rk * 128;
  if (!encode_bf16_planar_map(&a.tm_qh, a.qh, (long long)p->B * p->Hq, Sp) ||
      !encode_bf16_planar_map(&a.tm_kh, a.kh, (long long)p->B * p->Hkv, Sp) ||
      !encode_bf16_planar_map(&a.tm_vh, a.vh, (long long)p->B * p->Hkv, Sp) ||
      !encode_bf16_tokens_map(&a.tm_do, p->d_o, p->B, p->S, p->Hq, p->layout))
    return BSC_ERR_CUDA;
  a.q8 = p->q;
  a.k8 = p->k;
  a.vtn = p->vtn;
  a.q_sc = p->q_sc;
  a.k_sc = p->k_sc;
  a.vtn_sc = p->vtn_sc;
  a.o = p->o;
  a.dO = p->d_o;
  a.lse = p->lse;
  a.dq = p->dq;
  a.dk = p->dk;
  a.dv = p->dv;
  a.Sp = Sp;
  a.dev_status = p->dev_status;
  a.limit_ns = (unsigned long long)(p->wait_timeout_ms ? p->wait_timeout_ms : 2000u) * 1000000ull;
  a.B = p->B;
  a.S = p->S;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.layout = p->layout;
  a.scale = p->softmax_scale;
  a.scale_log2e = (float)((double)p->softmax_scale * 1.4426950408889634);
  return from_cuda(bsc::launch_attn_bwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

bsc_status bsc_read_device_status(const int32_t* dev_status, bsc_stream_t stream) {
  if (!dev_status) return BSC_ERR_NULL;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost, reinterpret_cast<cudaStream_t>(stream)) !=
          cudaSuccess ||
      cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BSC_ERR_CUDA;
  return v == 0 ? BSC_OK : BSC_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
