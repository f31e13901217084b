/*
 * bsc.h - C ABI of the leak-free causal MXFP8 attention forward library (libbsc.so, sm_103a).
 *
 * The operation: "[PyTorch] Add causal MXFP8 attention without future-token leakage through V
 * scales" (TransformerEngine PR #3865), Description.  A columnwise MXFP8 V scale is shared by 32
 * consecutive tokens, so under an ordinary causal mask a later token of a query's own 32-token
 * block can change how earlier visible V values round.  The method attends keys of completed
 * 32-token blocks (j < 32*floor(i/32)) in MXFP8 with the columnwise V, attends the query's own
 * block (at most 32 keys, j <= i) on a token-normalised V copy (one power-of-two amplitude per
 * token), and merges the two partials through their log-sum-exps, so output row i never depends
 * on a token after i.
 *
 * Conventions for every call:
 *   - Every buffer is device memory owned by the caller.  The library never allocates, frees or
 *     synchronises; all work is enqueued on `stream` (NULL = the legacy default stream).
 *   - Arguments are checked before anything is enqueued; on any error nothing is launched.
 *   - Calls hold no state between invocations and may be made from several host threads.
 *   - Tokens S must be a multiple of 32 (whole MX blocks) and D must be 128.  B, S or H equal to 0
 *     is an empty problem: the call returns BSC_OK and launches nothing (pointers are not
 *     inspected).
 *   - Every pointer must be 16-byte aligned.
 *   - The current CUDA device must be compute capability 10.3 (GB300).
 *   - Inputs are assumed finite; a NaN/Inf V value in a later token can reach earlier rows
 *     through a 0 * NaN product inside the diagonal key tile.
 *
 * Data layouts (BSHD: [B][S][H][D]; SBHD: [S][B][H][D]; D fastest in both).  Every scale array is
 * compact, in the operation's natural order (no padding, no swizzle):
 *   x_bf16, v_bf16, o_bf16    bf16 in the given layout
 *   x_e4m3, vtn_e4m3          E4M3 bytes, same layout and strides as the bf16 input
 *   v_e4m3_t                  E4M3 bytes of V transposed, [B][H][D][S] (tokens in order)
 *   x_sc (Q, K and MXFP8 O)   one scale byte per (b, h, s, 32-element block c = d/32):
 *                             [B][H][S][D/32], byte ((b*H + h)*S + s)*4 + c
 *   v_sc                      one scale byte per (b, h, 32-token block, d):
 *                             [B][H][S/32][D], byte ((b*H + h)*(S/32) + s/32)*D + d
 *   vtn_sc                    one token amplitude per (b, h, s): [B][H][S], byte (b*H + h)*S + s
 *   lse                       fp32 [B][Hq][S], natural log
 * Scale bytes are E8M0: value 2^(byte-127), 0xFF = NaN.  The attention kernels permute scales
 * into the tensor cores' scale-factor order themselves.
 *
 * Quantisation rule (OCP MX, E4M3 elements): for a block with maximum magnitude amax, the scale
 * byte is clamp(floor(log2 amax) - 8 + 127, 0, 254) (0 for amax = 0); each element is x*2^-e
 * rounded to nearest even on the E4M3 grid and saturated to +-448; a block holding NaN/Inf gets
 * scale 0xFF and element bytes 0x7F.
 */
#ifndef BSC_H
#define BSC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stream handle: a cudaStream_t. */
typedef struct CUstream_st* bsc_stream_t;

typedef enum {
  BSC_OK = 0,
  BSC_ERR_NULL = 1,           /* a required pointer is NULL */
  BSC_ERR_SHAPE = 2,          /* negative size, Hq not a multiple of Hkv, bad layout code */
  BSC_ERR_ALIGN = 3,          /* a pointer is not 16-byte aligned */
  BSC_ERR_UNSUPPORTED = 4,    /* D != 128, S % 32 != 0, wrong device, unsupported option */
  BSC_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed (launch, tensor map) */
  BSC_ERR_DEVICE_TIMEOUT = 6  /* a device-side wait gave up (see bsc_read_device_status) */
} bsc_status;

typedef enum { BSC_BSHD = 0, BSC_SBHD = 1 } bsc_layout;

/* Version of this ABI (bumped on any incompatible change). */
int bsc_abi_version(void);

/* Human-readable name of a status code (static storage). */
const char* bsc_status_string(bsc_status s);

/*
 * Rowwise MXFP8 quantisation of Q or K: one E8M0 scale per 32 consecutive elements along D of
 * each (b, s, h) row ("Q/K decoded from their rowwise MXFP8 bytes", PR #3865 Description).
 *   x_bf16 [in]  bf16 in `layout`;  x_e4m3 [out] same layout;  x_sc [out] [B][H][S][D/32].
 */
bsc_status mxfp8_quantize_qk_rowwise(const void* x_bf16, int B, int S, int H, int D, bsc_layout layout,
                                     uint8_t* x_e4m3, uint8_t* x_sc, bsc_stream_t stream);

/*
 * Columnwise MXFP8 quantisation of V: one E8M0 scale per 32 consecutive tokens of each (b, h, d)
 * ("A columnwise MXFP8 V scale is shared by 32 consecutive tokens", PR #3865 Description).
 *   v_bf16 [in] bf16 in `layout`;  v_e4m3_t [out] [B][H][D][S];  v_sc [out] [B][H][S/32][D].
 */
bsc_status mxfp8_quantize_v_colwise(const void* v_bf16, int B, int S, int H, int D, bsc_layout layout,
                                    uint8_t* v_e4m3_t, uint8_t* v_sc, bsc_stream_t stream);

/*
 * Token-normalised V copy: one power-of-two amplitude per (b, s, h) token row ("a
 * token-normalized copy of V (one power-of-two amplitude per token)", PR #3865 Description),
 * chosen by the same MX rule with the block spanning all D elements of the row.
 *   v_bf16 [in];  vtn_e4m3 [out] same layout as V;  vtn_sc [out] B*H*S bytes.
 */
bsc_status v_token_normalize(const void* v_bf16, int B, int S, int H, int D, bsc_layout layout,
                             uint8_t* vtn_e4m3, uint8_t* vtn_sc, bsc_stream_t stream);

/* Both V quantisations in one pass over V (one read); outputs as in the two calls above. */
bsc_status mxfp8_quantize_v_fused(const void* v_bf16, int B, int S, int H, int D, bsc_layout layout,
                                  uint8_t* v_e4m3_t, uint8_t* v_sc, uint8_t* vtn_e4m3, uint8_t* vtn_sc,
                                  bsc_stream_t stream);

/*
 * Scale rule of the quantisers.  FLOOR, used by every call above, is the OCP MX rule stated at
 * the top of this file.  CEIL rounds the scale up instead, e = ceil(log2(amax / 448)): the
 * smallest scale at which no element of the block saturates, one more than FLOOR exactly when
 * the significand of amax is above 1.75.  The pages say only that TE's MXFP8 attention reused
 * TE's existing quantisation kernels (PR #3865, base change list); CEIL is the "amax / scale
 * <= 448" reading of such a kernel, offered as a variant.
 */
typedef enum { BSC_SCALE_FLOOR = 0, BSC_SCALE_CEIL = 1 } bsc_scale_rule;
typedef enum {
  BSC_QUANT_ROWWISE = 0,      /* as mxfp8_quantize_qk_rowwise: x -> e4m3, sc */
  BSC_QUANT_V_COLWISE = 1,    /* as mxfp8_quantize_v_colwise: x -> e4m3 (the v_e4m3_t), sc */
  BSC_QUANT_V_TOKEN_NORM = 2, /* as v_token_normalize: x -> vtn_e4m3, vtn_sc */
  BSC_QUANT_V_FUSED = 3       /* as mxfp8_quantize_v_fused: all four outputs */
} bsc_quant_kind;
typedef struct {
  int kind;               /* bsc_quant_kind */
  const void* x;          /* [in] bf16 in `layout` */
  int B, S, H, D;
  int layout;             /* bsc_layout */
  int rule;               /* bsc_scale_rule */
  uint8_t* e4m3;          /* [out] rowwise bytes, or V columnwise bytes [B][H][D][S] */
  uint8_t* sc;            /* [out] [B][H][S][D/32] (rowwise) or [B][H][S/32][D] (V columnwise) */
  uint8_t* vtn_e4m3;      /* [out] token-normalised V bytes (token-norm and fused kinds) */
  uint8_t* vtn_sc;        /* [out] token amplitudes (token-norm and fused kinds) */
} bsc_quant_params;

/* Any of the four quantisations above with a chosen scale rule; layouts, sizes, ownership and
 * errors as in the matching call.  An unknown kind or rule is BSC_ERR_UNSUPPORTED. */
bsc_status mxfp8_quantize(const bsc_quant_params* p, bsc_stream_t stream);

/*
 * Every operand of the attention forward quantised in one launch: Q and K rowwise (as
 * mxfp8_quantize_qk_rowwise), V columnwise and token-normalised (as mxfp8_quantize_v_fused), each
 * tensor read once.  Outputs are byte-identical to those calls.  The pages quantise the three
 * operands in a separate step ahead of the attention and count it, with the launches, in a fixed
 * cost of about 1 ms at batch 1 (PR #3865, Performance); one launch for all three is this
 * library's form of that step.
 *   q [in] bf16 B x S x Hq x D in `layout`;  k, v [in] bf16 with Hkv heads;  Hq % Hkv == 0.
 *   q_e4m3, q_sc, k_e4m3, k_sc [out] as mxfp8_quantize_qk_rowwise for Q and K.
 *   v_e4m3_t, v_sc [out] as mxfp8_quantize_v_colwise; vtn_e4m3, vtn_sc [out] as v_token_normalize.
 *   Either V pair may be NULL (both pointers of the pair), not both.
 *   rule: bsc_scale_rule.  Errors as the calls above; an unknown rule is BSC_ERR_UNSUPPORTED.
 */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  int B, S, Hq, Hkv, D;
  int layout;             /* bsc_layout */
  int rule;               /* bsc_scale_rule */
  uint8_t* q_e4m3;
  uint8_t* q_sc;
  uint8_t* k_e4m3;
  uint8_t* k_sc;
  uint8_t* v_e4m3_t;
  uint8_t* v_sc;
  uint8_t* vtn_e4m3;
  uint8_t* vtn_sc;
} bsc_qkv_quant_params;
bsc_status mxfp8_quantize_qkv(const bsc_qkv_quant_params* p, bsc_stream_t stream);

typedef struct {
  const uint8_t* q;       /* [in] Q E4M3 bytes, `layout`, Hq heads */
  const uint8_t* q_sc;    /* [in] Q scales [B][Hq][S][D/32] */
  const uint8_t* k;       /* [in] K E4M3 bytes, `layout`, Hkv heads */
  const uint8_t* k_sc;    /* [in] K scales [B][Hkv][S][D/32] */
  const uint8_t* v_t;     /* [in] V columnwise E4M3 bytes, [B][Hkv][D][S] */
  const uint8_t* v_sc;    /* [in] V columnwise scales [B][Hkv][S/32][D] */
  const uint8_t* vtn;     /* [in] token-normalised V bytes, `layout` (unused when leaky = 1) */
  const uint8_t* vtn_sc;  /* [in] token amplitudes [B][Hkv][S] (unused when leaky = 1) */
  void* o;                /* [out] bf16 O in `layout`, Hq heads (may be NULL when o_e4m3 is set) */
  float* lse;             /* [out] [B][Hq][S], ln sum_{j<=i} exp(softmax_scale * q_i . k_j) */
  int B, S, Hq, Hkv, D;
  int layout;             /* bsc_layout */
  float softmax_scale;    /* finite and > 0, else BSC_ERR_UNSUPPORTED */
  /* Number of E4M3 terms P is split into for the MXFP8 P.V of completed blocks (1 or 2).  Each
   * row's weights are quantised per 32-key block with a power-of-two scale chosen from that row's
   * own scores in that block (the block's largest weight lands in [128, 256)), so a scale never
   * depends on another row or on a key the row cannot see.  The second term is the E4M3 residual
   * at the same scale.  The own block is one BF16 term. */
  int p_terms;
  /* 0: the method.  1: ordinary (leaky) causal MXFP8 - the own block is attended with the
   * columnwise V as well; a control that shows the leak. */
  int leaky;
  /* Optional device int32 (may be NULL).  Left untouched on success; a device-side wait that
   * gives up writes 0x100 | site.  Clear it before the call when you intend to read it. */
  int32_t* dev_status;
  /* Wall-clock limit of any single device-side wait, milliseconds (0 = 2000). */
  uint32_t wait_timeout_ms;
  /* Test hook: 1 makes the MMA issuer wait on a barrier nothing arrives on, so the call ends
   * through the wait limit with dev_status set.  Must be 0 in normal use. */
  int debug_stall;
  /* Optional MXFP8 O ("FROST SDPA fp8: block-scaled O epilogues (NVFP4 / MXFP8) with an sf_o
   * output", cudnn-frontend PR #1088 and its follow-up #1180, Summary: FP8_E4M3 O with one UE8M0
   * scale per 32 head-dim elements; that page keeps the scales in its swizzled atom order, this
   * library in the compact order of Q's scales).  When o_e4m3 is not NULL the epilogue also
   * writes O as E4M3 bytes in `layout` (Hq heads) and
   * o_sc [B][Hq][S][D/32] like Q's scales, by the quantisation rule above applied to the fp32 O
   * before any BF16 rounding.  o_sc is required with o_e4m3. */
  uint8_t* o_e4m3;
  uint8_t* o_sc;
} bsc_attn_fwd_params;

/*
 * Leak-free causal MXFP8 attention forward (PR #3865 Description: completed-block MXFP8 part,
 * own-block part on the token-normalised V, log-sum-exp merge).  GQA: query head h reads
 * KV head h / (Hq/Hkv).  Returns BF16 O and/or MXFP8 O, and fp32 LSE.
 * Causality: for finite inputs, row i of every output is bit-for-bit independent of the tokens
 * after i.  V must be finite for that to hold inside a 128-token tile: the diagonal tile's MMAs
 * multiply the zero weights of a row's later keys with those keys' V, and 0 x NaN (or 0 x the NaN
 * that a non-finite V block encodes to) is NaN, so a non-finite V element of token j makes the
 * earlier rows of j's 128-token tile non-finite.  Rows of earlier tiles never read token j.
 */
bsc_status mxfp8_causal_attn_fwd(const bsc_attn_fwd_params* p, bsc_stream_t stream);

typedef struct {
  const uint8_t* q;       /* [in] Q E4M3 bytes, `layout`, Hq heads */
  const uint8_t* q_sc;    /* [in] Q scales [B][Hq][S][D/32] */
  const uint8_t* k;       /* [in] K E4M3 bytes, `layout`, Hkv heads */
  const uint8_t* k_sc;    /* [in] K scales [B][Hkv][S][D/32] */
  const uint8_t* vtn;     /* [in] token-normalised V bytes, `layout`, Hkv heads */
  const uint8_t* vtn_sc;  /* [in] token amplitudes [B][Hkv][S] */
  const void* o;          /* [in] bf16 O of the forward, `layout`, Hq heads */
  const float* lse;       /* [in] LSE of the forward, [B][Hq][S], natural log */
  const void* d_o;        /* [in] bf16 dO, `layout`, Hq heads */
  void* dq;               /* [out] bf16, `layout`, Hq heads */
  void* dk;               /* [out] bf16, `layout`, Hkv heads */
  void* dv;               /* [out] bf16, `layout`, Hkv heads */
  int B, S, Hq, Hkv, D;
  int layout;             /* bsc_layout */
  float softmax_scale;    /* finite and > 0, else BSC_ERR_UNSUPPORTED */
  int32_t* dev_status;    /* optional, as in bsc_attn_fwd_params */
  uint32_t wait_timeout_ms;
  /* [scratch] device memory of at least bf16_attn_bwd_workspace_bytes(B, S, Hq, Hkv) bytes,
   * 16-byte aligned, overlapping no other argument; owned by the caller, contents on entry
   * ignored, on return undefined.  The call first writes there, once, what both backward kernels
   * read: Qh, Kh and the token-normalised Vt decoded to BF16 (one plane per batch and head, rows
   * padded to a multiple of 128 with zeros) and the per-row statistics Dlt_i and LSE_i*log2(e).
   * NULL: BSC_ERR_NULL; workspace_bytes below the required size: BSC_ERR_SHAPE. */
  float* workspace;
  size_t workspace_bytes;
} bsc_attn_bwd_params;

/*
 * Backward of the leak-free attention on decoded operands ("[PyTorch] Add causal MXFP8 attention
 * without future-token leakage through V scales", PR #3865, Description, Backward: an FP16/BF16
 * backward on Q and K decoded from their rowwise MXFP8 bytes and V decoded from the
 * token-normalised copy, so no gradient depends on a future token).  With s = scale*Qh.Kh^T on
 * keys j <= i: P = exp(s - LSE), dV = P^T dO, dP = dO.Vt^T, Dlt_i = <dO_i, O_i>,
 * dS = P*(dP - Dlt), dQ = scale*dS.Kh, dK = scale*dS^T.Qh; GQA: dK, dV of a KV head sum over
 * the query heads that read it.  BF16 tensor-core MMAs (P and dS rounded to BF16), fp32
 * accumulation, BF16 outputs.  Uses no memory beyond its arguments and the caller's workspace.
 */
bsc_status bf16_attn_bwd(const bsc_attn_bwd_params* p, bsc_stream_t stream);

/*
 * Bytes of workspace bf16_attn_bwd needs: B * Sp * (8 * Hq + 256 * (Hq + 2 * Hkv)) with
 * Sp = 128 * ceil(S / 128) (fp32 statistics per query row, a BF16 row of D = 128 per query and
 * per key and value row); 0 if a size is not positive.  Host only, no CUDA call.
 */
size_t bf16_attn_bwd_workspace_bytes(int B, int S, int Hq, int Hkv);

/*
 * The backward of bf16_attn_bwd without caller scratch: `workspace` and `workspace_bytes` of *p are
 * ignored and the call uses a fixed device array of this library (bf16_attn_bwd_static_capacity()
 * bytes, taken when the library's module holding it is loaded), so it allocates nothing.  The
 * pages have no counterpart of this call; it is a packaging of the same computation.  The array is
 * shared by every call on a device: calls must not overlap in time (one stream, or synchronised).
 * A call that needs more than the capacity: BSC_ERR_SHAPE, nothing launched.  Other arguments and
 * errors as bf16_attn_bwd.
 */
bsc_status bf16_attn_bwd_static(const bsc_attn_bwd_params* p, bsc_stream_t stream);

/* Bytes of the fixed workspace of bf16_attn_bwd_static.  Host only, no CUDA call. */
size_t bf16_attn_bwd_static_capacity(void);

/*
 * Synchronises `stream`, reads the int32 at `dev_status` and returns BSC_OK (0) or
 * BSC_ERR_DEVICE_TIMEOUT (non-zero).  The only call that synchronises.
 */
bsc_status bsc_read_device_status(const int32_t* dev_status, bsc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BSC_H */
