/*
 * mikv.h - C ABI of libmikv.so, the GB300 (sm_103a) hot path of MiKV, the
 * importance-aware mixed-precision KV cache ("No Token Left Behind: Reliable KV
 * Cache Compression via Importance-Aware Mixed Precision Quantization", arXiv
 * 2402.18096), with the optional CriticalKV two-stage selection (arXiv
 * 2502.03805).
 *
 * Sources cited below:
 *   [notes]      "No Token Left Behind" reading notes (velog.io), sections
 *                "Observation", "Key contributions 1)-3)", "3.4 Accelerating the
 *                Mixed-Precision KV Cache".
 *   [paperlayer] paperlayer.ai summary of arXiv 2402.18096v1, sections 3.1-3.4,
 *                4.1, 5, Appendix C.
 *   [criticalkv] gist.science summary of arXiv 2502.03805 (CriticalKV),
 *                "Theoretical framework" and "Algorithm: perturbation-constrained
 *                selection".
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every array pointer is a DEVICE pointer owned by the caller.  The library
 *   never allocates device memory; scratch comes from a caller workspace whose
 *   size a *_workspace_bytes query returns.
 * - fp16 arrays are passed as uint16_t* holding IEEE binary16 bit patterns.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Calls are asynchronous on that stream; none synchronises the host.
 * - All shapes are row-major, innermost dimension last, contiguous.
 * - Return value: MIKV_OK (0) or a negative status.  On any error nothing is
 *   launched and nothing is written; mikv_last_error() returns a message
 *   (thread-local, valid until the next call on the same thread).
 * - Head dimension D must be 128 (the kernels are specialised for it); the
 *   quantisation group is gs = D/2 = 64 ([notes] "2) Outlier-aware": group size
 *   = half the attention head dimension, against RoPE artefacts).
 * - GQA: Hq query heads, Hkv key/value heads, rep = Hq/Hkv in 1..8; query head
 *   h reads key head h / rep.
 */
#ifndef MIKV_H_
#define MIKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define MIKV_OK 0
#define MIKV_EINVAL (-1)       /* null pointer where one is required, bad enum, bad scalar */
#define MIKV_ESHAPE (-2)       /* dimension, capacity or count out of range */
#define MIKV_EALIGN (-3)       /* a buffer is not 16-byte aligned */
#define MIKV_EUNSUPPORTED (-4) /* bit width or head dimension the kernels do not implement */
#define MIKV_ECUDA (-5)        /* a CUDA launch failed (message in mikv_last_error) */

/* mikv_score_update modes */
#define MIKV_PREFILL 0
#define MIKV_DECODE 1

/* mikv_select policies */
#define MIKV_H2O 0
#define MIKV_CRITICALKV 1
#define MIKV_DEMOTE 2

/* mikv_quantize_append tiers */
#define MIKV_TIER_HI 0
#define MIKV_TIER_LO 1
#define MIKV_TIER_DEMOTE 2

/* mikv_cache.key_mode: how the low tier stores keys */
#define MIKV_KEYS_PER_TOKEN 0   /* per-token asymmetric groups of 64 channels (MiKV) */
#define MIKV_KEYS_PER_CHANNEL 1 /* per-channel groups of 64 slots (the Appendix C alternative) */

/*
 * One layer's two-tier cache ([notes] "Key contributions 1)" and "3)": tokens
 * an eviction policy would drop are kept in low precision next to the important
 * tokens kept in FP16 or INT8; [notes] 3.4: after positional embedding
 * attention is permutation invariant, so each precision lives in its own
 * contiguous tier).  Counts are uniform over (batch, key head).
 *
 * Slot layouts (all per [B][Hkv][capacity]):
 *   hi_bits == 16: k_hi, v_hi fp16 [B][Hkv][cap_hi][D]; hi meta unused (NULL).
 *   hi_bits == 8 or 4: k_hi, v_hi uint8 codes [B][Hkv][cap_hi][D*hi_bits/8],
 *                  packed as the lo tier below; k_hi_meta, v_hi_meta
 *                  [B][Hkv][cap_hi][D/64][2] fp16 (scale, zero).  An INT4 important
 *                  tier with an INT2 low tier is the INT4/INT2 split of the pages'
 *                  precision sweeps ([notes] "3)", [paperlayer] 4.1).
 *   lo tier:       k_lo, v_lo uint8 [B][Hkv][cap_lo][D*lo_bits/8] packed codes:
 *                  channel c sits in bits [(c*lo_bits) % 8, +lo_bits) of byte
 *                  (c*lo_bits)/8, least significant bits first;
 *                  k_lo_meta, v_lo_meta [B][Hkv][cap_lo][D/64][2] fp16 (scale, zero).
 *   pos_hi, pos_lo int32: original sequence position of each slot.
 *   scores         fp32 [B][Hkv][cap_hi]: accumulated H2O importance of each hi slot.
 *   balancer       fp32 [B][Hkv][D] or NULL (identity).
 * lo_bits <= hi_bits.  Quantised keys (INT8/INT4 hi tier and the lo tier) hold I(k*b); the FP16 tier holds
 * the original k.  Values are never balanced.
 * Code and meta buffers must be 16-byte aligned.
 *
 * key_mode == MIKV_KEYS_PER_CHANNEL ([notes] Appendix C remarks: per-channel quantisation
 * isolates outlier channels, but a cache then has to hold KV pairs in a buffer until enough
 * have accumulated; [paperlayer] C: group size 64, keys per channel, 20 % FP16 / 80 % INTx):
 *   hi_bits must be 16 and lo_bits 2 or 4; cap_lo a multiple of 64; the balancer is not used.
 *   The low tier's slots [0, n_lo - n_lo % 64) form closed groups of 64 slots: k_lo holds
 *   per-token code rows as above, but their scale and zero are per (group, channel):
 *   k_lo_meta [B][Hkv][cap_lo/64][D][2] fp16 (scale, zero), the per-token quantizer's rule
 *   applied to each channel's 64 values; v_lo and v_lo_meta stay per token.
 *   The last n_lo % 64 retained pairs wait unquantised:
 *   k_pend, v_pend fp16 [B][Hkv][64][D], row p = slot n_lo - n_lo % 64 + p (pos_lo holds their
 *   positions).  The pair that brings them to 64 closes the group: its keys are quantised per
 *   channel and its values per token into the group's slots.  Attention reads closed groups
 *   and waiting pairs (as stored); waiting pairs are attended with the original q.
 * key_mode == MIKV_KEYS_PER_TOKEN (0): k_pend, v_pend unused (NULL).
 */
typedef struct mikv_cache {
  int32_t B, Hkv, Hq, D;
  int32_t hi_bits, lo_bits; /* hi in {16, 8, 4}; lo in {2, 4, 8}, lo <= hi */
  int32_t cap_hi, cap_lo;
  int32_t n_hi, n_lo; /* current counts; updated on the host by the calls that change them */
  void* k_hi;
  void* v_hi;
  void* k_hi_meta;
  void* v_hi_meta;
  void* k_lo;
  void* v_lo;
  void* k_lo_meta;
  void* v_lo_meta;
  int32_t* pos_hi;
  int32_t* pos_lo;
  const float* balancer;
  float* scores;
  int32_t key_mode; /* MIKV_KEYS_PER_TOKEN or MIKV_KEYS_PER_CHANNEL */
  void* k_pend;     /* per-channel keys: waiting pairs, fp16 [B][Hkv][64][D] */
  void* v_pend;
} mikv_cache;

/*
 * Channel balancer ([notes] "2) Outlier-aware", balancer equation; [paperlayer]
 * 3.2): b[b][g][c] = sqrt(Mq / Mk), Mq = max over the group's query heads and
 * the T prompt tokens of |q[b][h][t][c]|, Mk = max over t of |k[b][g][t][c]|;
 * b = 1 where Mq or Mk is 0.  The ratio and the square root are fp32,
 * round-to-nearest-even.  q, k are the post-RoPE prompt tensors.
 *   q    fp16 [B][Hq][T][D]      k fp16 [B][Hkv][T][D]
 *   b_out fp32 [B][Hkv][D]       (written)
 *   ws   >= mikv_balance_workspace_bytes(B, Hkv, D) bytes, 16-byte aligned
 * Errors: EINVAL (null), ESHAPE (T < 1, Hq % Hkv, rep > 8), EUNSUPPORTED (D != 128),
 * EALIGN, ECUDA.
 */
int mikv_balance_prefill(const uint16_t* q, const uint16_t* k, int B, int Hq, int Hkv, int T,
                         int D, float* b_out, void* ws, size_t ws_bytes, void* stream);
size_t mikv_balance_workspace_bytes(int B, int Hkv, int D);

/*
 * Allocation-free variant of mikv_balance_prefill (the paper has no counterpart:
 * this is a deployment convenience).  Same inputs, output and result, but no
 * workspace argument: the scratch lives in a static device array inside the
 * library.  It is meant for callers that cannot allocate device memory, such as
 * a plugin that its host framework hands only input and output buffers, or a
 * serving loop that must never enter the allocator (cudaMalloc/cudaFree
 * synchronise the device and may fail under memory pressure).
 *   Limit: B * Hkv <= 1024 (the array holds 2 x 1024 x 128 floats, 1 MiB, on
 *   every device that loads the library, until the process exits); larger
 *   shapes return MIKV_ESHAPE.
 *   Every call looks up that array's device address in the context current on
 *   the calling thread (a lookup, not an allocation), so the address stays right
 *   after cudaDeviceReset or under another context.  The first call on a device
 *   may load the library's device code there; make it before any stream capture.
 *   All calls share the one array and each clears it first: calls whose kernels
 *   can overlap on the GPU (different streams, without ordering) race and
 *   return wrong results.  Calls allocate nothing.
 * Errors: as mikv_balance_prefill, plus ESHAPE above the limit and ECUDA if the
 * array's address cannot be obtained.
 */
int mikv_balance_prefill_noalloc(const uint16_t* q, const uint16_t* k, int B, int Hq, int Hkv,
                                 int T, int D, float* b_out, void* stream);

/*
 * H2O importance ([notes] "Observation 1-4" and "Key contributions 1)": H2O,
 * accumulated attention; read as the plain H2O definition).
 * MIKV_PREFILL: column sums of the causal softmax over the T prompt rows,
 *   S^h[b][h][i] = sum_{t >= i} exp(q_t.k_i/sqrt(D) - lse_t), and the group sum
 *   S[b][g][i] = sum over the group's query heads, h ascending, fp32.
 *   Uses q fp16 [B][Hq][T][D], k fp16 [B][Hkv][T][D] and the dims of c
 *   (c->B, Hkv, Hq, D; no cache buffer is touched).
 *   scores_full fp32 [B][Hkv][T] (written); scores_head fp32 [B][Hq][T] (written if not NULL).
 *   ws >= mikv_score_workspace_bytes(B, Hq, T) bytes.
 * MIKV_DECODE: c->scores[b][g][j] += sum_h exp(hi_logits[b][h][j] - lse[b][h]) for
 *   every hi slot j < c->n_hi; hi_logits fp32 [B][Hq][cap_hi] and lse fp32 [B][Hq]
 *   as written by mikv_decode_attention.  q, k, T, scores_*, ws unused.
 * Errors: EINVAL, ESHAPE, EUNSUPPORTED, ECUDA.
 */
int mikv_score_update(int mode, const uint16_t* q, const uint16_t* k, int T,
                      const float* hi_logits, const float* lse, mikv_cache* c,
                      float* scores_full, float* scores_head, void* ws, size_t ws_bytes,
                      void* stream);
size_t mikv_score_workspace_bytes(int B, int Hq, int T);

/*
 * Selection.  Budget n_keep(L) = min(L, max(window, floor(budget_pct*L/100))):
 * the `window` most recent positions are always kept and count inside the
 * budget ([paperlayer] 5: local tokens and heavy hitters).  Ranking key
 * (score descending, position ascending); ties keep the lower position.
 * MIKV_H2O ([notes] "Key contributions 1)"): keep the window plus the top
 *   n_keep - window older tokens by scores [B][Hkv][L].
 * MIKV_CRITICALKV ([criticalkv] "Algorithm"): bud = n_keep - window,
 *   b' = floor(alpha*bud), b'' = bud - b'; stage 1 takes the top b' older tokens
 *   by scores; stage 2 takes the top b'' of the remaining older tokens by
 *   C_i = sum_h fl(S^h_i * N[b][h][i]) (fp32, h ascending over the group), with
 *   S^h = scores_head [B][Hq][L] and N the projected-value L1 norms
 *   ([criticalkv] "Theoretical framework": V W_O):
 *     N[b][h][i] = || v[b][h/rep][i][:] . w_o[h*D:(h+1)*D][:] ||_1.
 *   If w_o != NULL, N is computed from v fp16 [B][Hkv][L][D] and w_o fp16
 *   [Hq*D][hidden] (hidden % 128 == 0) and written to vwo_norm fp32 [B][Hq][L];
 *   if w_o == NULL, vwo_norm is read as given.
 * Outputs (H2O, CRITICALKV): keep_pos int32 [B][Hkv][n_keep] ascending,
 *   evict_pos int32 [B][Hkv][L - n_keep] ascending, keep_scores fp32
 *   [B][Hkv][n_keep] = scores at keep_pos (written if not NULL).
 * MIKV_DEMOTE: reads c->scores, c->pos_hi and c->n_hi; among hi slots with
 *   pos < L - window picks the minimum of (score ascending, position descending)
 *   and writes its slot index to evict_pos [B][Hkv]; L is the current length.
 *   Requires c->n_hi > window.
 * ws >= mikv_select_workspace_bytes(policy, B, Hkv, Hq, L, hidden), 16-byte aligned;
 *   CRITICALKV keeps the stage-2 keys there and, when w_o != NULL, a transposed copy of
 *   w_o ([hidden][Hq*D] fp16, so both tensor-core operands are channel-contiguous).
 * Errors: EINVAL (null, policy, alpha outside [0,1]), ESHAPE (L, budget, window,
 * hidden, B*Hkv*L >= 2^31), EALIGN (v, w_o, ws), EUNSUPPORTED, ECUDA.
 */
int mikv_select(int policy, const mikv_cache* c, int L, int budget_pct, int window, float alpha,
                const float* scores, const float* scores_head, const uint16_t* v,
                const uint16_t* w_o, int hidden, float* vwo_norm, int32_t* keep_pos,
                int32_t* evict_pos, float* keep_scores, void* ws, size_t ws_bytes, void* stream);
size_t mikv_select_workspace_bytes(int policy, int B, int Hkv, int Hq, int L, int hidden);

/*
 * Quantise-and-append ([notes] "Key contributions 1)": per-token asymmetric
 * quantisation (LLM-QAT) of the retained tokens; "2)": keys as I(k*b);
 * "3)": INT8 important tier).  Per token, key head and 64-channel group:
 *   x = fl(k*b) for keys of a quantised tier, x = v for values;
 *   s = fp16(fl(max-min)/qmax), z = fp16(min),
 *   code = clamp(rint_even(fl(fl(x - z)/s)), 0, qmax), code 0 where s == 0.
 * MIKV_TIER_HI: slots n_hi..n_hi+n_tokens-1 take source tokens src_pos
 *   [B][Hkv][n_tokens] (indices into k, v fp16 [B][Hkv][src_len][D]); FP16
 *   tier: copy; INT8 tier: quantise.  pos_hi = src_pos + pos_base;
 *   scores = src_scores [B][Hkv][n_tokens] if not NULL, else 0.  n_hi += n_tokens.
 * MIKV_TIER_LO: same into the lo tier (lo_bits); pos_lo = src_pos + pos_base.
 *   n_lo += n_tokens.
 * MIKV_TIER_DEMOTE: n_tokens must be 1; src_pos [B][Hkv] are hi slots.  Each is
 *   re-quantised into lo slot n_lo from what the hi tier holds (FP16: fl(k*b)
 *   and v; INT8: fl(fl(s*code)+z), already balanced); then the last hi slot
 *   (k, v, meta, pos, score) moves into the freed slot.  n_hi -= 1, n_lo += 1.
 *   k, v, src_len, pos_base, src_scores unused.
 * Per-channel keys (c->key_mode == MIKV_KEYS_PER_CHANNEL): MIKV_TIER_LO requires n_lo % 64 == 0;
 *   the first floor(n_tokens / 64) * 64 tokens close groups at once (keys per channel, values
 *   per token), the rest wait in k_pend / v_pend.  MIKV_TIER_DEMOTE moves the victim's FP16
 *   pair into the waiting buffer (no quantisation); when it is the 64th waiting pair, a second
 *   launch closes the group.  MIKV_TIER_HI is unchanged (FP16 copy).
 * Counts in *c are updated on the host after a successful launch.
 * Errors: EINVAL, ESHAPE (capacity overflow, src_len, a per-channel LO append off a group
 * boundary), EALIGN, EUNSUPPORTED, ECUDA.
 */
int mikv_quantize_append(int tier, const uint16_t* k, const uint16_t* v, int src_len,
                         const int32_t* src_pos, int n_tokens, int pos_base,
                         const float* src_scores, mikv_cache* c, void* stream);

/*
 * Decode attention over the two-tier cache ([notes] 3.4 and [paperlayer] 3.4:
 * tiers grouped by precision, K and V low precision, Q and the attention map
 * floating point; [notes] "2)": quantised keys are attended with q/b).
 * For query head h of key head g:
 *   FP16 hi tier:  logit = q_h . k / sqrt(D)        (original q and k)
 *   quantised tiers: logit = (q_h / b_g) . k~ / sqrt(D)   (k~ dequantised k*b)
 *   p = softmax over both tiers; out_h = sum p v~; lse_h = log sum exp(logit).
 *   q      fp16 [B][Hq][D]
 *   out    fp32 [B][Hq][D]; lse fp32 [B][Hq] (natural log)
 *   hi_logits fp32 [B][Hq][cap_hi] (slots < n_hi written) or NULL
 *   ws >= mikv_decode_workspace_bytes(c) bytes (split-K partial results and the
 *   per-(batch, key head) query fragments).
 * Per-channel keys: closed groups give logit = (q_h . (s (.) code + z)) / sqrt(D) with the
 *   group's per-channel scale s and zero z (no balancer); waiting pairs are attended as FP16
 *   with the original q, like the FP16 tier.  The workspace also holds the fp32 query.
 * Requires n_hi + n_lo >= 1.  Errors: EINVAL, ESHAPE, EALIGN, EUNSUPPORTED, ECUDA.
 */
int mikv_decode_attention(const uint16_t* q, const mikv_cache* c, float* out, float* lse,
                          float* hi_logits, void* ws, size_t ws_bytes, void* stream);
size_t mikv_decode_workspace_bytes(const mikv_cache* c);

/*
 * One whole decode step in four launches (the same arithmetic as the sequence
 * quantize_append(HI) -> decode_attention -> score_update(DECODE) ->
 * select(DEMOTE) -> quantize_append(DEMOTE), with identical results):
 *   1. the new token (k_new, v_new fp16 [B][Hkv][D], position `pos`) is appended
 *      to the important tier with score 0 (the same launch prepares the query);
 *   2. q fp16 [B][Hq][D] attends over both tiers (split-K partials);
 *   3. the partials are merged into out fp32 [B][Hq][D] and lse fp32 [B][Hq];
 *   4. the step's attention is added to the H2O score of every important slot,
 *      and, if policy == MIKV_H2O and the important tier now holds more than
 *      n_keep(pos + 1) tokens, the victim (see mikv_select(MIKV_DEMOTE)) is
 *      demoted.  MIKV_CRITICALKV never demotes.
 * The order follows H2O: evict after the step's attention ([notes] "Key
 * contributions 1)"; [paperlayer] 5).  Per-channel keys: the demoted pair joins the waiting
 * buffer, and a fifth launch closes its group when it is the 64th.  ws >= mikv_decode_step_workspace_bytes(c)
 * (partials, the important-tier logits, per-chunk victim candidates).  Counts in
 * *c are updated.  Two calls must not share a workspace concurrently.
 * Errors: EINVAL, ESHAPE (capacity, budget, workspace), EALIGN, EUNSUPPORTED
 * (cap_hi above 65535*1024), ECUDA.
 */
int mikv_decode_step(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new, int pos,
                     int budget_pct, int window, int policy, mikv_cache* c, float* out, float* lse,
                     void* ws, size_t ws_bytes, void* stream);
size_t mikv_decode_step_workspace_bytes(const mikv_cache* c);

/*
 * K9: the step after attention ([criticalkv] "Theoretical framework": the output
 * perturbation L = ||o - o^||_1 of replacing the full cache, bounded through the value
 * states projected by W_O; "Experimental results": reported per attention head).
 * Head h reaches the hidden state through rows h*D .. h*D + D - 1 of W_O:
 *   y[b][:]  = sum_h o[b][h][:] . W_O^(h)                      (the output projection)
 *   pert[b][h] = || (o[b][h][:] - o_hat[b][h][:]) . W_O^(h) ||_1  (sum over hidden)
 * o, o_hat fp32 [B][Hq][D] (D = 128): e.g. decode attention over the full cache and over
 * the mixed-precision (or evicted) cache.  w_o_t fp16 [hidden][Hq*D], row-major: W_O
 * transposed, the layout nn.Linear stores; hidden % 128 == 0; 16-byte aligned.
 * y fp32 [B][hidden] is written if not NULL; pert fp32 [B][Hq] if not
 * NULL (needs o_hat).  With w_o_t == NULL, pert[b][h] = || o - o_hat ||_1 over D (y must
 * be NULL).  Products are formed from fp16 (hi, lo) splits of o and o - o_hat with fp32
 * accumulation (relative error ~1e-6).
 * ws >= mikv_output_perturbation_workspace_bytes(B, Hq, hidden), 16-byte aligned
 * (operand tiles and per-column partial sums).  Stream-ordered; no synchronisation.
 * Errors: EINVAL (null o, pert without o_hat, y without w_o_t, null ws), EUNSUPPORTED (D),
 * ESHAPE (B < 1, Hq outside 1..128, hidden, workspace), EALIGN, ECUDA.
 */
int mikv_output_perturbation(const float* o, const float* o_hat, const uint16_t* w_o_t, int B, int Hq,
                             int D, int hidden, float* y, float* pert, void* ws, size_t ws_bytes,
                             void* stream);
size_t mikv_output_perturbation_workspace_bytes(int B, int Hq, int hidden);

/*
 * Post-attention top-k over the full cache ([notes] "1-4) Quantitative analysis": the
 * oracle-eviction simulation computes the attention map over the full cache first and
 * applies top-k sparsity after the attention, an upper-bound proxy for eviction).
 * c must hold the full cache in its FP16 tier (hi_bits 16, n_lo 0, n_hi = L >= 1 tokens,
 * e.g. a prefill at budget 100).  Per (batch, query head) the k = max(1, floor(p*L/100))
 * largest logits q.k/sqrt(D) are kept (ties to the lower slot) and
 *   out[b][h] = sum_{i kept} exp(l_i - m) v_i / sum_{i kept} exp(l_i - m),
 *   lse[b][h] = log sum_{i kept} exp(l_i)            (natural log; written if not NULL),
 *   keep_idx [B][Hq][k] int32 = the kept slots, ascending (written if not NULL).
 * q fp16 [B][Hq][D]; out fp32 [B][Hq][D].  Three stages, stream-ordered: the decode attention
 * of this cache (all logits), a radix select per head, attention over the kept slots.
 * ws >= mikv_topk_attention_workspace_bytes(c, budget_pct), 16-byte aligned.
 * Errors: EINVAL (null), EUNSUPPORTED (not a full FP16 cache), ESHAPE (budget, heads,
 * n_hi outside 1..131072, workspace), and those of mikv_decode_attention.
 */
int mikv_topk_attention(const uint16_t* q, const mikv_cache* c, int budget_pct, float* out, float* lse,
                        int32_t* keep_idx, void* ws, size_t ws_bytes, void* stream);
size_t mikv_topk_attention_workspace_bytes(const mikv_cache* c, int budget_pct);

/*
 * Per-channel group quantisation of retained-tier keys ([notes] Appendix C remarks;
 * [paperlayer] C: group size 64, keys quantised per channel), standalone: the arithmetic the
 * per-channel cache (mikv_cache.key_mode) applies when it closes a group.
 * k fp16 [units][n][D] (D = 128): each unit's keys in slot order.  The floor(n / 64) full
 * groups are quantised; the n mod 64 keys after them are left alone (they wait in FP16 until
 * a group is full).  Per (group, channel c), over the group's 64 values of channel c:
 *   s = fp16(fl(fl(mx - mn) / qmax)), z = fp16(mn),
 *   code = clamp(rint_even(fl(fl(x - z) / s)), 0, qmax), 0 where s == 0.
 * codes uint8 [units][n][D*bits/8]: per-token rows (channel c at bits (c*bits) mod 8 of byte
 * c*bits/8, LSB first), rows of full groups written; meta fp16 [units][n/64][D][2] =
 * (scale, zero).  bits in {2, 4, 8}.  Stream-ordered.
 * Errors: EINVAL (null), EUNSUPPORTED (D, bits), ESHAPE (units outside 1..65535, n < 0).
 */
int mikv_channel_quantize(const uint16_t* k, int units, int n, int D, int bits, uint8_t* codes,
                          uint16_t* meta, void* stream);

/*
 * Measurement hook (no counterpart in the papers): while set, every
 * mikv_decode_attention and mikv_decode_step call made by this thread records
 * `begin` (a cudaEvent_t) on its stream just before the split-K attention
 * launch and `end` just after it, so that a caller can time that kernel alone
 * with cudaEventElapsedTime.  The events are owned by the caller and must stay
 * valid while set; (NULL, NULL) clears the hook.  Setting only one of the two
 * is EINVAL.  A failed record is reported as ECUDA by the call that made it.
 */
int mikv_set_attention_events(void* begin, void* end);

/*
 * Wait status of the tensor-core kernels (no counterpart in the papers; a failure report).
 * The tcgen05 kernels (K3's two prefill score passes in mikv_score_update(MIKV_PREFILL),
 * K6's V.W_O norms in mikv_select(MIKV_CRITICALKV) with w_o, K9 in
 * mikv_output_perturbation) hand tiles between a TMA/MMA thread and their consumer warps
 * through mbarriers, and every wait there gives up after ~4 million polls instead of
 * spinning for ever.  No wait is expected to run out; if one does, the thread that gave up
 * issues no further copy or MMA, its later waits poll only ~1000 times each (so a stuck
 * pipeline still ends in a bounded time, and what was issued before has that long to land),
 * the kernel writes NaN into the outputs of the affected CTA (prefill scores and -lse rows,
 * V.W_O norms, perturbation and y partial sums) and sets a bit in a device-side status word.
 * The call that launched it has already returned MIKV_OK (launches are asynchronous).
 * mikv_wait_status stores the OR of the bits set since the last clear in *bits:
 *   1 = K3 pass 1 (row log-sum-exp), 2 = K3 pass 2 (column sums), 4 = K6 (V.W_O norms),
 *   8 = K9 (output perturbation), 16 = mikv_wait_probe
 * and clears them if `clear` is non-zero.  It copies synchronously: call it after the work
 * in question has completed (e.g. after synchronising its stream).
 * Errors: EINVAL (null bits), ECUDA (the copy failed).
 */
int mikv_wait_status(unsigned* bits, int clear);

/*
 * Self-check of the give-up path above (no counterpart in the papers): one thread waits, with
 * the same bounded wait as the tensor-core kernels, on an mbarrier of one arrival that it
 * makes itself only if `arrive` is non-zero.  Without the arrival the first wait gives up
 * after `polls` polls (1 .. 2^24), a second one after the short limit, and status bit 16 is
 * set; with it nothing is set.  No memory is read or written but that bit; the launch does
 * not disturb the context.  Stream-ordered.  Errors: EINVAL (polls), ECUDA (launch).
 */
int mikv_wait_probe(int64_t polls, int arrive, void* stream);

/* Message of the last failed call on this thread ("" if none). */
const char* mikv_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MIKV_H_ */
