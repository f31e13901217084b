// Internal launch interface shared by the C-ABI layer and the kernels (not part of the ABI).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsc {

// rule: 0 = OCP floor scale rule, 1 = ceil (no element saturates)
cudaError_t launch_quant_rowwise(const void* x, uint8_t* q, uint8_t* sc, int B, int S, int H, int layout,
                                 cudaStream_t st, int rule = 0);
// Q and K rowwise and V (columnwise and/or token-normalised) in one launch.
struct QkvQuantArgs {
  const void* q;
  const void* k;
  const void* v;
  int B, S, Hq, Hkv, layout, rule;
  uint8_t* q8;
  uint8_t* q_sc;
  uint8_t* k8;
  uint8_t* k_sc;
  uint8_t* vt;       // may be nullptr (no columnwise copy)
  uint8_t* vsc;
  uint8_t* vtn;      // may be nullptr (no token-normalised copy)
  uint8_t* vtn_sc;
  long long nv_blocks, nq_blocks;   // set by the launcher
};
cudaError_t launch_quant_qkv(QkvQuantArgs a, cudaStream_t st);
cudaError_t launch_quant_v(const void* v, uint8_t* vt, uint8_t* vsc, uint8_t* vtn, uint8_t* vtn_sc, int B, int S,
                           int H, int layout, cudaStream_t st, int rule = 0);

// Everything the attention kernel reads, by value (tensor maps must be 64-byte aligned).
struct AttnArgs {
  CUtensorMap tm_q;     // Q bytes, 4-D {D, Hq, S, B}, box {128,1,128,1}, 128-byte swizzle
  CUtensorMap tm_k;     // K bytes, 4-D {D, Hkv, S, B}, same box
  CUtensorMap tm_v;     // V columnwise bytes, 2-D {S, B*Hkv*D}, box {128,128}, 128-byte swizzle
  const uint8_t* q_sc;     // compact [B][Hq][S][4]
  const uint8_t* k_sc;     // compact [B][Hkv][S][4]
  const uint8_t* v_sc;     // compact [B][Hkv][S/32][128]
  const uint8_t* vtn;      // token-normalised V bytes, K's layout (unused when leaky)
  const uint8_t* vtn_sc;   // [B][Hkv][S]
  void* o;              // bf16 O, or nullptr
  uint8_t* o8;          // E4M3 O, or nullptr
  uint8_t* o_sc;        // compact [B][Hq][S][4] scales of the E4M3 O (with o8)
  float* lse;
  int32_t* dev_status;
  unsigned long long limit_ns;
  int B, S, Hq, Hkv, layout;
  float scale_log2e;
  int p_terms;
  int leaky;
  int inject_stall;
};

cudaError_t launch_attn_fwd(const AttnArgs& args, cudaStream_t st);

// Arguments of the backward kernels (prep, dQ, and dK/dV).
struct BwdArgs {
  CUtensorMap tm_qh;    // decoded Q, BF16 workspace planes [B*Hq][Sp][D], box {64,128,1}, 128-byte swizzle
  CUtensorMap tm_kh;    // decoded K, [B*Hkv][Sp][D], likewise
  CUtensorMap tm_vh;    // decoded token-normalised V, [B*Hkv][Sp][D], likewise
  CUtensorMap tm_do;    // dO bf16, 4-D {D, Hq, S, B}, box {64,1,128,1}, 128-byte swizzle
  const uint8_t* q8;    // Q bytes, `layout`, Hq heads
  const uint8_t* k8;    // K bytes, `layout`, Hkv heads
  const uint8_t* vtn;   // token-normalised V bytes, `layout`, Hkv heads
  const uint8_t* q_sc;  // compact [B][Hq][S][4]
  const uint8_t* k_sc;  // compact [B][Hkv][S][4]
  const uint8_t* vtn_sc;  // [B][Hkv][S]
  const void* o;        // bf16 O of the forward, Q's layout
  const void* dO;       // bf16 dO, Q's layout
  const float* lse;     // [B][Hq][S], natural log
  void* dq;             // bf16, Q's layout
  void* dk;             // bf16, K's layout
  void* dv;             // bf16, K's layout
  float* ws;            // workspace: Dlt [B][Hq][Sp], then LSE * log2(e) [B][Hq][Sp]
  uint16_t* qh;         // workspace: the BF16 planes behind tm_qh, tm_kh, tm_vh
  uint16_t* kh;
  uint16_t* vh;
  int32_t* dev_status;
  unsigned long long limit_ns;
  int B, S, Hq, Hkv, layout;
  int Sp;               // S rounded up to the 128-row tile
  float scale, scale_log2e;
};

// Workspace bytes of the backward: the statistics (2 x 4 B per query row) and the BF16 planes of
// Qh, Kh and Vt (256 B per row), rows padded to Sp.
size_t bwd_workspace_bytes(int B, int S, int Hq, int Hkv);

cudaError_t launch_attn_bwd(const BwdArgs& args, cudaStream_t st);

}  // namespace bsc
