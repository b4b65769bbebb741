/*
 * engram.h -- C ABI of the Engram lookup layer (hashed n-gram conditional
 * memory) for one NVIDIA GB300 GPU (sm_103a).
 *
 * Pages cited by title:
 *   [P-V41]    "DeepSeek-V4.1 模型结构（5）：记忆，Engram"
 *   [P-LMNT]   "Engram条件记忆：DeepSeek-V4.1-Flash中196B稀疏参数N-gram哈希查表的实现原理"
 *   [P-O1]     "条件记忆：DeepSeek V4.1 Engram 如何用 O(1) 查表换掉一层计算"
 *   [P-DS4]    "ds4.c 学习笔记" -- glossary entry "Engram"
 *   [P-DETAIL] "DeepSeek Engram 详解：把静态知识从计算里拆出来"
 *
 * Conventions shared by every entry point
 *   - Every function returns 0 (ENGRAM_OK) or a negative ENGRAM_E_* code and
 *     never throws.  engram_last_error() returns a thread-local message for
 *     the last failure on the calling thread.
 *   - Pointers named *_d are device pointers; the caller allocates and owns
 *     them.  The library allocates no device memory.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  Results are visible after
 *     the caller synchronises that stream.
 *   - Problems found on the device (bad token id, row out of range, bad
 *     history slot, a bounded wait that ran out) are OR-ed into the caller's
 *     device word `status_d` (ENGRAM_ST_* bits) when it is non-NULL; the
 *     kernel then writes a defined fallback (masked position / zero row) and
 *     completes.  No kernel traps.
 *   - bf16 tensors are passed as uint16_t* holding bf16 bit patterns.
 *   - Every kernel is compiled for sm_103a only; entry points that launch
 *     work return ENGRAM_E_DEVICE on any other GPU.
 */
#ifndef ENGRAM_H
#define ENGRAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ENGRAM_ABI_VERSION 3

#define ENGRAM_MAX_LAYERS 8
#define ENGRAM_MAX_NGRAM 4   /* n-gram orders 2..max_ngram; history depth max_ngram-1 */
#define ENGRAM_MAX_COLS 32   /* (max_ngram-1) * n_heads */
#define ENGRAM_DEAD (-1)     /* raw / compressed id of an image position */
#define ENGRAM_ROW_BYTES 264 /* 256 E4M3 weights + 8 E8M0 scales */
#define ENGRAM_HEAD_DIM 256

/* Return codes. */
enum {
  ENGRAM_OK = 0,
  ENGRAM_E_INVALID = -1,  /* null pointer, bad count, bad layer index */
  ENGRAM_E_VOCAB = -2,    /* compressed vocabulary differs from the expected one */
  ENGRAM_E_SHAPE = -3,    /* unsupported or inconsistent sizes */
  ENGRAM_E_ALIGN = -4,    /* a pointer is not aligned as the entry point requires */
  ENGRAM_E_RANGE = -5,    /* a value does not fit (row count >= 2^31, multiplier bound) */
  ENGRAM_E_CUDA = -6,     /* a CUDA runtime call or launch failed */
  ENGRAM_E_DEVICE = -7    /* the current device is not an sm_103 GPU */
};

/* Bits OR-ed into the device status word. */
#define ENGRAM_ST_BAD_TOKEN 0x1u /* raw id not in [0, V_raw) and not DEAD, or map value not in [0, V) */
#define ENGRAM_ST_BAD_ROW 0x2u   /* row id not in [0, total_rows) */
#define ENGRAM_ST_BAD_SLOT 0x4u  /* decode history slot >= n_slots */
#define ENGRAM_ST_TIMEOUT 0x8u   /* a bounded on-chip wait ran out; outputs are undefined */

/* ------------------------------------------------------------------------ */
/* Layout                                                                    */
/* ------------------------------------------------------------------------ */

/* Inputs of engram_build_layout.  The names follow the checkpoint config
 * keys listed on [P-LMNT] (整体架构 table): engram_vocab_size (base_rows),
 * engram_layer_ids, engram_max_ngram_size, engram_n_heads, engram_head_dim,
 * engram_compressed_vocab_size (vocab_compressed). */
typedef struct engram_layout_params {
  int64_t vocab_compressed;  /* V: compressed vocabulary size */
  int64_t expected_vocab;    /* 0: no check; otherwise must equal V (ENGRAM_E_VOCAB) */
  int64_t base_rows;         /* primes are taken strictly above this value */
  int32_t n_layers;          /* 1..ENGRAM_MAX_LAYERS */
  int32_t layer_ids[ENGRAM_MAX_LAYERS];
  int32_t max_ngram;         /* 2..ENGRAM_MAX_NGRAM (4 in DeepSeek-V4.1) */
  int32_t n_heads;           /* heads per order (8); (max_ngram-1)*n_heads <= ENGRAM_MAX_COLS */
  int32_t head_dim;          /* 256 (the only row format supported) */
  int32_t pad_id;            /* compressed id used for padding, 0 <= pad_id < V */
  int32_t use_multiplier_override; /* nonzero: take multipliers from the array below */
  int64_t multiplier_override[ENGRAM_MAX_LAYERS][ENGRAM_MAX_NGRAM];
} engram_layout_params;

/* Immutable description of every layer's table.  Column j (0 <= j < n_cols)
 * is order n = 2 + j / n_heads, head k = j % n_heads. */
typedef struct engram_layout {
  int64_t vocab_compressed;
  int64_t base_rows;
  int32_t n_layers;
  int32_t max_ngram;
  int32_t n_heads;
  int32_t n_cols;
  int32_t head_dim;
  int32_t pad_id;
  int32_t layer_ids[ENGRAM_MAX_LAYERS];
  int64_t total_rows[ENGRAM_MAX_LAYERS];               /* sum of the layer's primes */
  int64_t primes[ENGRAM_MAX_LAYERS][ENGRAM_MAX_COLS];
  int64_t offsets[ENGRAM_MAX_LAYERS][ENGRAM_MAX_COLS]; /* exclusive cumulative sum */
  uint64_t reciprocal[ENGRAM_MAX_LAYERS][ENGRAM_MAX_COLS]; /* floor((2^64-1)/p), for the modulo */
  int64_t multipliers[ENGRAM_MAX_LAYERS][ENGRAM_MAX_NGRAM];
} engram_layout;

/* Build the table layout on the host (no device work).
 *
 * Primes: [P-V41] §"一层只有一张表" (search upward from engram_vocab_size,
 * one prime per head, never reused; the printed per-layer min/max/sum for
 * layers 1 and 14) and [P-O1] §2.2 (one ascending sequence consumed in
 * (layer, order, head) order; primality by deterministic Miller-Rabin).
 * The library takes the primes strictly greater than base_rows.
 * Offsets: [P-O1] §2.2 / [P-DS4] §布局与哈希探测 step 3 (cumulative sum).
 * Multipliers: [P-V41] §"哈希函数" under eq. (H) and [P-O1] §4.3 -- per
 * layer, odd, drawn from a generator seeded with 10007 * layer_id and bounded
 * by int64max // V // 2.  This library draws them from SplitMix64 (Steele,
 * Lea & Flood 2014): r_i = i-th output mod half, m_i = 2 r_i + 1, with
 * half = ((2^63-1) // V) // 2.  Checkpoint multipliers from another generator
 * are passed through use_multiplier_override (each must be odd and keep
 * (V-1) * m within int64).
 *
 * Errors: ENGRAM_E_INVALID (null pointer, counts out of range, pad id not a
 * compressed id), ENGRAM_E_VOCAB (expected_vocab != V, the guard of
 * [P-V41] under eq. (H) and [P-O1] §2.1), ENGRAM_E_SHAPE (head_dim != 256,
 * too many columns), ENGRAM_E_RANGE (a layer's row count would reach 2^31, or
 * an override multiplier breaks the bound). */
int engram_build_layout(const engram_layout_params* params, engram_layout* out);

/* sizeof(engram_layout_params) and sizeof(engram_layout), for bindings. */
size_t engram_layout_params_size(void);
size_t engram_layout_size(void);

/* ------------------------------------------------------------------------ */
/* Hash (stages 1-3): token map, suffix window, multiplicative-XOR mix,      */
/* per-head prime modulo plus segment offset.                                */
/* ------------------------------------------------------------------------ */

/* Prefill hash over packed sequences.
 *
 * For every position t of sequence s (positions cu_seqlens_d[s] ..
 * cu_seqlens_d[s+1]-1):
 *   x'_t = token_map_d[raw_ids_d[t]]                 ([P-V41] §tokenizer 压缩)
 *   g_i  = x'_{t-i} for i < max_ngram; before the sequence start the slot comes
 *          from hist_d[s][i-1-(t-start)] (most recent first) or, with
 *          hist_d == NULL, is pad_id                  ([P-DETAIL] §3.2)
 *   from the first DEAD slot on every slot is pad_id ([P-V41] image tokens,
 *          [P-LMNT] §多模态细节)
 *   mix_n = XOR_{i<n} g_i * m_i, n = 2..max_ngram   ([P-V41] eq. (H))
 *   row_ids_d[t][j] = mix_{n(j)} mod p_j + offset_j  ([P-DS4] step 3)
 *   mask_d[t] = 1 if the position itself is DEAD, else 0.
 * After the hash, hist_d (if non-NULL) is advanced to the last max_ngram-1
 * compressed ids of each sequence (DEAD kept as -1), so a later call on the
 * next chunk continues the same n-grams ([P-LMNT] §第二步: prefill and decode
 * share one history).
 *
 * Arguments
 *   layout, layer     layout from engram_build_layout; 0 <= layer < n_layers
 *   raw_ids_d         int32 [n_tokens]; values in [0, vocab_raw) or DEAD
 *   cu_seqlens_d      int64 [n_seqs+1], nondecreasing, [0] = 0, [n_seqs] = n_tokens
 *   token_map_d       int32 [vocab_raw]; values in [0, V)
 *   hist_d            int32 [n_seqs][max_ngram-1] in/out, or NULL (all pad, not written)
 *   row_ids_d         int32 [n_tokens][n_cols] out
 *   mask_d            uint8 [n_tokens] out
 *   status_d          int32 device word (OR-ed ENGRAM_ST_*), or NULL
 * A bad raw id or map value sets ENGRAM_ST_BAD_TOKEN and the position is
 * treated as DEAD.  n_tokens == 0 is a no-op. */
int engram_hash(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                int64_t n_tokens, const int64_t* cu_seqlens_d, int32_t n_seqs,
                const int32_t* token_map_d, int64_t vocab_raw, int32_t* hist_d,
                int32_t* row_ids_d, uint8_t* mask_d, int32_t* status_d, void* stream);

/* engram_hash for every layer of the layout in one launch ([P-O1] §2.4: the
 * row ids depend only on the token ids, so serving code hashes all Engram
 * layers before the layer loop).  The window and the history are shared by
 * the layers; row_ids_d is int32 [n_layers][n_tokens][n_cols] (layer-major),
 * mask_d and hist_d as engram_hash (hist_d advanced once). */
int engram_hash_all_layers(const engram_layout* layout, const int32_t* raw_ids_d, int64_t n_tokens,
                           const int64_t* cu_seqlens_d, int32_t n_seqs, const int32_t* token_map_d,
                           int64_t vocab_raw, int32_t* hist_d, int32_t* row_ids_d, uint8_t* mask_d,
                           int32_t* status_d, void* stream);

/* One decode step: one new raw id per batch entry, hashed against the
 * sequence's rolling history and committed in the same launch ([P-O1] §4.4;
 * [P-DS4] §布局与哈希探测: the hash state is the last 3 ids and a copy of it is
 * a snapshot).
 *
 *   raw_ids_d  int32 [batch]
 *   slots_d    int32 [batch]: history row of each entry, or -1 for a padding
 *              entry (hashed with an all-pad history, masked, commits nothing;
 *              [P-O1] §4.4: padding rows must not pollute the history).
 *              Two entries of one call must not name the same slot.
 *   hist_d     int32 [n_slots][max_ngram-1] in/out; a used slot becomes
 *              (x', h0, h1, ...) after the step.
 *   row_ids_d  int32 [batch][n_cols]; mask_d uint8 [batch] (1 = DEAD or padding)
 * A slot >= n_slots sets ENGRAM_ST_BAD_SLOT and the entry is treated as padding. */
int engram_hash_step(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                     const int32_t* slots_d, int32_t batch, const int32_t* token_map_d,
                     int64_t vocab_raw, int32_t* hist_d, int64_t n_slots, int32_t* row_ids_d,
                     uint8_t* mask_d, int32_t* status_d, void* stream);

/* ------------------------------------------------------------------------ */
/* Gather + dequantise (stage 4)                                             */
/* ------------------------------------------------------------------------ */

/* e_d[t][256*j + c] = bf16_rne(E4M3(b[c]) * 2^(s[c/32] - 127)) where b, s are
 * the 256 weight bytes and 8 scale bytes of row row_ids_d[t][j]
 * ([P-V41] §"196B 参数怎么存、怎么取"; [P-DS4] §布局与哈希探测 and the
 * e4m3_e8m0_32_row264 encoding of §永不常驻的 I/O 设计; [P-O1] §2.3).
 * E4M3 is OCP FP8 E4M3 (no infinities, 0x7F/0xFF NaN), E8M0 is the OCP scale
 * (0xFF NaN).  The result is the exact product rounded once to bf16.
 *
 *   table_d      uint8 [total_rows][264], 16-byte aligned (ENGRAM_E_ALIGN);
 *                device memory, or pinned / ATS-visible host memory that the
 *                kernel reads over NVLink-C2C
 *   table_bytes  size of the table allocation in bytes, >= total_rows * 264
 *   row_ids_d    int32 [n_tokens][n_cols], or NULL for the ids t*n_cols + j
 *   e_d          bf16 [n_tokens][n_cols*256] out, 16-byte aligned
 * A row id outside [0, total_rows) sets ENGRAM_ST_BAD_ROW and its 256 outputs
 * are +0. */
int engram_gather_dequant(const uint8_t* table_d, int64_t total_rows, int64_t table_bytes,
                          const int32_t* row_ids_d, int64_t n_tokens, int32_t n_cols,
                          uint16_t* e_d, int32_t* status_d, void* stream);

/* Stages 1-4 fused: the prefill hash of engram_hash and the gather of
 * engram_gather_dequant in one kernel.  The warp that gathers a position's
 * rows computes their ids from the position's token window, so the ids need
 * not round-trip through memory ([P-O1] §2.4: the rows depend only on the
 * token ids).  Arguments as in engram_hash and engram_gather_dequant, with
 * the table of layer `layer` (total_rows from the layout):
 *   table_d      uint8 [total_rows][264], 16-byte aligned; table_bytes >= total_rows * 264
 *   e_d          bf16 [n_tokens][n_cols*256] out, 16-byte aligned
 *   mask_d       uint8 [n_tokens] out (1 = DEAD position)
 *   row_ids_d    int32 [n_tokens][n_cols] out, or NULL (not written)
 *   hist_d       int32 [n_seqs][max_ngram-1] in/out carried history, or NULL
 * The history is advanced by a second launch after every position has read
 * it.  Status bits as for the two calls it fuses. */
int engram_hash_gather(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d, int64_t n_tokens,
                       const int64_t* cu_seqlens_d, int32_t n_seqs, const int32_t* token_map_d, int64_t vocab_raw,
                       int32_t* hist_d, const uint8_t* table_d, int64_t table_bytes, uint16_t* e_d,
                       uint8_t* mask_d, int32_t* row_ids_d, int32_t* status_d, void* stream);

/* The gather for the block-scaled FP8 projection: the rows are copied as
 * stored instead of dequantised ([P-O1] §2.3: E4M3 payload with E8M0 scales
 * per 32 elements).  With T128 = n_tokens rounded up to a multiple of 128 and
 * P(t) = (t & ~127) | ((t & 31) << 2) | ((t >> 5) & 3), for position t and
 * column j:
 *   e8_d[t][256 j + c]                  = weight byte c of row row_ids_d[t][j]
 *   sf_d[(2 j + b / 4) * T128 + P(t)], byte b % 4 = scale byte b of that row
 * i.e. the scales are grouped per 128-element k-block, one 32-bit word of four
 * E8M0 scales per (k-block, position), and within each 128 positions the word
 * of position p0 + r + 32 c sits at p0 + 4 r + c: the 512-byte image the FP8
 * projection copies into tensor memory as it is (tcgen05.cp).  Positions
 * n_tokens .. T128-1 get scale words 0x7F7F7F7F.  A row id outside [0,
 * total_rows) sets ENGRAM_ST_BAD_ROW and gives zero bytes with scales 127
 * (the value 0).
 *   e8_d  uint8 [n_tokens][n_cols*256], 16-byte aligned
 *   sf_d  uint32 [n_cols*2][T128], 16-byte aligned */
int engram_gather_fp8(const uint8_t* table_d, int64_t total_rows, int64_t table_bytes, const int32_t* row_ids_d,
                      int64_t n_tokens, int32_t n_cols, uint8_t* e8_d, uint32_t* sf_d, int32_t* status_d,
                      void* stream);

/* engram_hash_gather with the FP8 outputs of engram_gather_fp8. */
int engram_hash_gather_fp8(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d, int64_t n_tokens,
                           const int64_t* cu_seqlens_d, int32_t n_seqs, const int32_t* token_map_d,
                           int64_t vocab_raw, int32_t* hist_d, const uint8_t* table_d, int64_t table_bytes,
                           uint8_t* e8_d, uint32_t* sf_d, uint8_t* mask_d, int32_t* row_ids_d, int32_t* status_d,
                           void* stream);

/* One decode step fused with its gather: the hash of engram_hash_step and
 * the gather of engram_gather_dequant in one kernel ([P-O1] §4.4: the decode
 * hash state is the last 3 ids of each sequence; [P-O1] §2.4: the rows depend
 * only on the token ids).  The warp that gathers entry b computes its row ids
 * from raw_ids_d[b] and the history row slots_d[b], then rolls that history
 * row; entries of one call must name distinct slots.  Arguments as in
 * engram_hash_step and engram_gather_dequant, with the table of layer `layer`:
 *   table_d    uint8 [total_rows][264], 16-byte aligned; table_bytes >= total_rows * 264
 *   e_d        bf16 [batch][n_cols*256] out, 16-byte aligned
 *   mask_d     uint8 [batch] out (1 = DEAD or padding entry)
 *   row_ids_d  int32 [batch][n_cols] out, or NULL (not written)
 * Status bits as for the two calls it fuses. */
int engram_hash_gather_step(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                            const int32_t* slots_d, int32_t batch, const int32_t* token_map_d, int64_t vocab_raw,
                            int32_t* hist_d, int64_t n_slots, const uint8_t* table_d, int64_t table_bytes,
                            uint16_t* e_d, uint8_t* mask_d, int32_t* row_ids_d, int32_t* status_d, void* stream);

/* engram_hash_gather_step with the FP8 outputs of engram_gather_fp8
 * (e8_d uint8 [batch][n_cols*256] 16-byte aligned, sf_d uint32
 * [n_cols*2][batch rounded up to 128] 16-byte aligned, in that call's order). */
int engram_hash_gather_step_fp8(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                                const int32_t* slots_d, int32_t batch, const int32_t* token_map_d,
                                int64_t vocab_raw, int32_t* hist_d, int64_t n_slots, const uint8_t* table_d,
                                int64_t table_bytes, uint8_t* e8_d, uint32_t* sf_d, uint8_t* mask_d,
                                int32_t* row_ids_d, int32_t* status_d, void* stream);

/* Stage 4 for a table of plain bf16 rows of any width (the generic-shape row
 * format: the Engram paper's 27B model reads 16 rows of 80 elements per
 * position into hidden 2560, [P-DETAIL] §5 after its worked example; the page
 * sizes that table at 2 bytes per element, §8.4).  Rows are copied as stored:
 *   e_d[t][j*row_dim + c] = table_d[row_ids_d[t][j]][c]
 *   table_d    bf16 [total_rows][row_dim], 16-byte aligned; row_dim a multiple
 *              of 8 in [8, 4096]
 *   row_ids_d  int32 [n_tokens][n_cols]
 *   e_d        bf16 [n_tokens][n_cols*row_dim] out, 16-byte aligned
 * A row id outside [0, total_rows) sets ENGRAM_ST_BAD_ROW and its row_dim
 * outputs are +0.  The projection takes e as is (K = n_cols*row_dim, a
 * multiple of 64). */
int engram_gather_rows_bf16(const uint16_t* table_d, int64_t total_rows, int32_t row_dim, const int32_t* row_ids_d,
                            int64_t n_tokens, int32_t n_cols, uint16_t* e_d, int32_t* status_d, void* stream);

/* Stages 1-4 fused for a bf16-row table: the hash of engram_hash_gather with
 * the copy of engram_gather_rows_bf16 (total_rows from the layout), then the
 * history commit.  Arguments and status bits as in those two calls. */
int engram_hash_gather_rows_bf16(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                                 int64_t n_tokens, const int64_t* cu_seqlens_d, int32_t n_seqs,
                                 const int32_t* token_map_d, int64_t vocab_raw, int32_t* hist_d,
                                 const uint16_t* table_d, int32_t row_dim, uint16_t* e_d, uint8_t* mask_d,
                                 int32_t* row_ids_d, int32_t* status_d, void* stream);

/* Dequantise rows that already sit contiguously in device memory (e.g. after
 * a host-side gather and one DMA): e_d[i/n_cols][256*(i%n_cols) + c] from
 * row i of rows_d, for i < n_rows (a multiple of n_cols).  Same arithmetic as
 * engram_gather_dequant.  rows_d is uint8 [n_rows][264], 16-byte aligned;
 * rows_bytes is its allocation size (>= n_rows * 264). */
int engram_dequant_rows(const uint8_t* rows_d, int64_t n_rows, int64_t rows_bytes, int32_t n_cols,
                        uint16_t* e_d, int32_t* status_d, void* stream);

/* ------------------------------------------------------------------------ */
/* Host-resident table (Grace memory)                                         */
/* ------------------------------------------------------------------------ */

/* The rows to fetch depend only on the token ids, so the table can live in
 * host memory and be fetched while earlier layers compute ([P-V41]
 * §"196B 参数怎么存、怎么取"; [P-O1] §4.1; [P-DETAIL] §8.2).  A pinned or
 * ATS-visible host table can be passed directly to engram_gather_dequant
 * (reads over NVLink-C2C).  Alternatively the rows are gathered by host
 * threads into a contiguous staging buffer, moved by one DMA and
 * dequantised with engram_dequant_rows:
 *
 * engram_host_gather copies row row_ids_h[i] of table_h (uint8 [total_rows]
 * [264], host) to staging_h + 264 i for i < n_rows, with n_threads OpenMP
 * threads (0: the OpenMP default).  Rows outside [0, total_rows) become 264
 * zero bytes (they dequantise to +0) and are counted in *bad_rows (nullable).
 * Runs on the calling thread; all pointers are host pointers. */
int engram_host_gather(const uint8_t* table_h, int64_t total_rows, const int32_t* row_ids_h, int64_t n_rows,
                       uint8_t* staging_h, int32_t n_threads, int64_t* bad_rows);

/* engram_host_gather enqueued on `stream` with cudaLaunchHostFunc: it runs
 * after the work already on the stream (for instance the device-to-host copy
 * of row_ids_h) and before the work enqueued later (the host-to-device copy of
 * staging_h), on CUDA's host-callback thread.  The buffers must stay valid
 * until the stream reaches it; *bad_rows is written before later stream work
 * starts (left untouched when n_rows == 0, which enqueues nothing). */
int engram_host_gather_async(const uint8_t* table_h, int64_t total_rows, const int32_t* row_ids_h,
                             int64_t n_rows, uint8_t* staging_h, int32_t n_threads, int64_t* bad_rows,
                             void* stream);

/* ------------------------------------------------------------------------ */
/* wkv projection with the gate reduction fused (stage 5a/5b)                */
/* ------------------------------------------------------------------------ */

/* Repack wkv from [K][N] (kv = e @ wkv, [P-V41] §"每条流一个 key 的设计":
 * one [6144, 25600] matrix) to the tiled K-major operand layout of the
 * tensor-core projection: [N/128][K/64][128][64], i.e. element (k, n) lands at
 * ((n/128 * K/64 + k/64) * 128 + n%128) * 64 + k%64, so every 128 x 64 operand
 * tile is 16 KB contiguous.  One-time, for static weights.  Both bf16, N*K
 * elements; requires K % 64 == 0 and N % 128 == 0 (ENGRAM_E_SHAPE). */
int engram_pack_wkv(const uint16_t* wkv_d, int64_t K, int64_t N, uint16_t* wkv_packed_d,
                    void* stream);

/* Bytes of the partial-sum buffer of engram_project:
 * float32 [n_tokens][hc][hidden/256][4]. */
size_t engram_project_partials_bytes(int64_t n_tokens, int32_t hidden, int32_t hc);

/* kv = e @ wkv on the tensor cores (bf16 x bf16 -> fp32), with the gate's
 * reductions in the epilogue ([P-V41] §门控; [P-DS4] §消费):
 *   columns [m*H, (m+1)*H) are key k^(m+1), m < hc; columns [hc*H, (hc+1)*H)
 *   are the value v.
 *   For every token t, stream m and 256-column tile q of key m the epilogue
 *   writes partials_d[t][m][q] = { sum_i h_{m,i} q_w[i][m] k_w[i][m] k_{m,i},
 *   sum_i k_{m,i}^2, sum_i h_{m,i}^2, 0 } over the tile's 256 columns i;
 *   keys are not stored.  The value is stored as v_d[t][i] = bf16_rne(v_i).
 *
 *   e_d          bf16 [n_tokens][K], K = n_cols*256, 16-byte aligned
 *   wkv_packed_d bf16, (hc+1)*hidden*K elements from engram_pack_wkv, 16-byte aligned
 *   h_d          bf16 [n_tokens][hc][hidden] residual streams (read only here)
 *   q_w_d, k_w_d float32 [hidden][hc]
 *   partials_d   float32, engram_project_partials_bytes(...) bytes
 *   v_d          bf16 [n_tokens][hidden] out
 * Requires hidden % 256 == 0, K % 64 == 0, 1 <= hc <= 8.  A bounded
 * on-chip wait that runs out sets ENGRAM_ST_TIMEOUT. */
int engram_project(const uint16_t* e_d, int64_t n_tokens, int64_t K, const uint16_t* wkv_packed_d,
                   int32_t hidden, int32_t hc, const uint16_t* h_d, const float* q_w_d,
                   const float* k_w_d, float* partials_d, uint16_t* v_d, int32_t* status_d,
                   void* stream);

/* ------------------------------------------------------------------------ */
/* Block-scaled FP8 projection (stage 5a on block-FP8 weights)               */
/* ------------------------------------------------------------------------ */

/* [P-O1] §2.3: the released model's projection weights are block-FP8.  Here
 * wkv is E4M3 codes w8_d uint8 [K][N] (kv = e @ wkv) with one E8M0 scale per
 * 32 consecutive rows of k in each column, sf_d uint8 [K/32][N]; value
 * E4M3(w) * 2^(s - 127).  engram_pack_wkv_fp8 repacks them once into the
 * operand layouts of the FP8 projection: w8_packed_d uint8, K*N bytes, tiles
 * [N/128][K/128][128][128] (element (k, n) at ((n/128 * K/128 + k/128) * 128
 * + n%128) * 128 + k%128); sf_packed_d uint32 [K/128][N], byte j of word
 * (kb, P(n)) = the scale of rows kb*128 + 32 j .. +31 of column n, with P the
 * order within each 128 columns of engram_gather_fp8's scales.  K and N
 * multiples of 128; sf_packed_d 16-byte aligned for the projection. */
int engram_pack_wkv_fp8(const uint8_t* w8_d, const uint8_t* sf_d, int64_t K, int64_t N, uint8_t* w8_packed_d,
                        uint32_t* sf_packed_d, void* stream);

/* engram_project on FP8 operands: e in the engram_gather_fp8 form (e8_d uint8
 * [n_tokens][K], sfa_d uint32 [K/128][T128], 16-byte aligned) and the packed
 * FP8 wkv.  The scale words travel with the operand tiles (TMA) and are
 * copied into tensor memory by the MMA-issuing thread (tcgen05.cp); the
 * tensor cores take the E4M3 values with their E8M0 scales (tcgen05.mma
 * kind::mxf8f6f4, block size 32) and accumulate in fp32; the outputs
 * (partials_d, v_d) are those of engram_project.  K % 128 == 0; other
 * requirements as for engram_project.  A bounded on-chip wait that runs out
 * sets ENGRAM_ST_TIMEOUT. */
int engram_project_fp8(const uint8_t* e8_d, const uint32_t* sfa_d, int64_t n_tokens, int64_t K,
                       const uint8_t* w8_packed_d, const uint32_t* sfb_d, int32_t hidden, int32_t hc,
                       const uint16_t* h_d, const float* q_w_d, const float* k_w_d, float* partials_d,
                       uint16_t* v_d, int32_t* status_d, void* stream);

/* engram_project_gate on FP8 operands (same workspace, engram_project_gate_workspace_bytes).
 * It runs engram_project_fp8 and engram_gate_add inside the workspace: the
 * FP8 kernel keeps one accumulator buffer, so a fused epilogue would not
 * overlap the next tile's main loop, and the two kernels are faster at every
 * size measured.  (engram_kernel_options.fp8_fused = 1 selects the fused
 * FP8 kernel above 1536 tokens, for comparisons.) */
int engram_project_gate_fp8(const uint8_t* e8_d, const uint32_t* sfa_d, int64_t n_tokens, int64_t K,
                            const uint8_t* w8_packed_d, const uint32_t* sfb_d, int32_t hidden, int32_t hc,
                            uint16_t* h_d, const float* q_w_d, const float* k_w_d, const uint8_t* mask_d, float eps,
                            float clamp, float score_scale, float* gate_out_d, void* workspace_d,
                            size_t workspace_bytes, int32_t* status_d, void* stream);

/* ------------------------------------------------------------------------ */
/* Gate + residual add (stage 5b/5c)                                          */
/* ------------------------------------------------------------------------ */

/* For every token t and stream m (sums over the partials' tiles in a fixed
 * order):
 *   s = dot * rsqrt(hh/H + eps) * rsqrt(kk/H + eps) * score_scale
 *   g = sigmoid(copysign(sqrt(max(|s|, clamp)), s))
 *   h_d[t][m][i] <- bf16_rne(h + g * bf16(v_d[t][i]))   in fp32
 * ([P-V41] §门控 and §"sigmoid 之前多一步带符号的平方根"; [P-DS4] §消费).
 * Masked positions (mask_d[t] != 0) leave h_d untouched and get g = 0
 * ([P-V41] image tokens; [P-DS4] step 4: the masked branch returns).
 * score_scale is H^-0.5, the reading of the pages the library follows ([P-V41]
 * derives s = sqrt(d) cos(theta); [P-DS4] prints a sqrt(width) factor).
 *
 *   partials_d   from engram_project
 *   v_d          bf16 [n_tokens][hidden]
 *   h_d          bf16 [n_tokens][hc][hidden], updated in place, 16-byte aligned
 *   mask_d       uint8 [n_tokens], or NULL (no masked positions)
 *   gate_out_d   float32 [n_tokens][hc] out, or NULL
 * With h_d = NULL only the gates are computed (gate_out_d required, v_d may
 * be NULL): the first half of the short-convolution variant below. */
int engram_gate_add(const float* partials_d, const uint16_t* v_d, uint16_t* h_d,
                    const uint8_t* mask_d, int64_t n_tokens, int32_t hidden, int32_t hc, float eps,
                    float clamp, float score_scale, float* gate_out_d, void* stream);

/* ------------------------------------------------------------------------ */
/* Short causal convolution (the original Engram layer's stage 5c)            */
/* ------------------------------------------------------------------------ */

/* The original Engram layer refines the gated value before the residual add
 * ([P-DETAIL] §4.2 and the pseudo code of §五; [P-V41] §"V4.1 相对原版的两处改动"
 * names it as the step V4.1 dropped).  For every position t of a sequence and
 * stream m, with V~ = g * bf16(v):
 *   n_t = gamma[m] * V~_t / sqrt(mean_i(V~_t,i^2) + eps)         (RMSNorm)
 *   c_t = sum_{k < kernel_size} w[k][m] * n_{t - k*dilation}     (depthwise, causal)
 *   h_d[t][m][i] <- bf16_rne(h + (V~_t,i + SiLU(c_t,i)))         in fp32
 * (gamma folded into the filter taps; SiLU with the fast exponential and
 * division, a few ulp plus about 1.2|c| ulp)
 * w[k] multiplies the value k*dilation positions back (a PyTorch Conv1d
 * filter W[ch][0][j] with left padding maps to w[k] = W[..][K-1-k]); there is
 * no bias.  The pages use kernel 4 with dilation = the largest n-gram order.
 * Masked positions have g = 0 (so V~ = 0 and n = 0) and still receive
 * SiLU(c_t) from earlier positions.
 *
 * Before a sequence start the filter reads zeros, or, with state_d, the
 * normalised values of the sequence's previous (kernel_size-1)*dilation
 * positions ([P-DETAIL] §9.5: 9 for kernel 4, dilation 3).  The state of slot
 * b is a ring: state_d[b][(p mod R)][m][i] holds n / gamma[m][i] (the RMS-
 * normalised value before the RMSNorm weight) of absolute position p,
 * R = (kernel_size-1)*dilation, and state_head_d[b] = (positions seen) mod R.
 * A new sequence starts from a zeroed ring and head 0.  The call reads the
 * old state, then writes the last min(R, len) values of every sequence and
 * advances its head.  Slots must be distinct within one call.
 *
 *   gate_d       float32 [n_tokens][hc] (engram_gate_add with h_d = NULL)
 *   v_d          bf16 [n_tokens][hidden] (engram_project), 16-byte aligned
 *   h_d          bf16 [n_tokens][hc][hidden], updated in place, 16-byte aligned
 *   mask_d       uint8 [n_tokens] or NULL
 *   cu_seqlens_d int64 [n_seqs+1] packed sequences, or NULL: every position is
 *                its own sequence (decode; n_seqs == n_tokens)
 *   slots_d      int32 [n_seqs] state slot per sequence, or NULL (slot = s);
 *                a negative slot is padding: its positions are untouched and
 *                it keeps no state; a slot >= n_slots (with a state) sets
 *                ENGRAM_ST_BAD_SLOT and is treated as padding
 *   conv_w_d     float32 [kernel_size][hc][hidden], 16-byte aligned
 *   gamma_d      float32 [hc][hidden], 16-byte aligned
 *   state_d      float32 [n_slots][R][hc][hidden] or NULL (zeros, no state kept)
 *   state_head_d int32 [n_slots]
 *   workspace_d  engram_short_conv_workspace_bytes(n_tokens, hc) bytes, 256-byte aligned
 * Requires hidden % 256 == 0, 1 <= hc <= 8, 1 <= kernel_size <= 4,
 * dilation >= 1 and R <= 64 (ENGRAM_E_SHAPE). */
size_t engram_short_conv_workspace_bytes(int64_t n_tokens, int32_t hc);
int engram_short_conv_add(const float* gate_d, const uint16_t* v_d, uint16_t* h_d, const uint8_t* mask_d,
                          int64_t n_tokens, int32_t hidden, int32_t hc, const int64_t* cu_seqlens_d,
                          int64_t n_seqs, const int32_t* slots_d, const float* conv_w_d, const float* gamma_d,
                          int32_t kernel_size, int32_t dilation, float eps, float* state_d,
                          int32_t* state_head_d, int64_t n_slots, void* workspace_d, size_t workspace_bytes,
                          int32_t* status_d, void* stream);

/* ------------------------------------------------------------------------ */
/* Projection with the gate and residual fused (stage 5a-5c in one kernel)    */
/* ------------------------------------------------------------------------ */

/* Bytes of the workspace of engram_project_gate: the partial sums
 * (engram_project_partials_bytes), then int32 counters
 * (2*ceil(n_tokens/256) * (4*hc + 1) + 1 words), then fp32 gates
 * (2*ceil(n_tokens/256) * 128 * hc), then bf16 v (n_tokens * hidden) for the
 * two-kernel path; each part on a 256-byte boundary. */
size_t engram_project_gate_workspace_bytes(int64_t n_tokens, int32_t hidden, int32_t hc);

/* The same result as engram_project followed by engram_gate_add, computed in
 * one cooperative tensor-core kernel ([P-V41] §门控; [P-DS4] §消费).  Key
 * tiles publish their partial sums; the epilogue warp that publishes the last
 * tile of a (128-row block, stream, 32-row quarter) sums that group's partials
 * in tile order and writes its gates; each value tile waits (bounded) for its
 * block's gates and applies h <- bf16(h + g * bf16(v)) directly, so v is never
 * stored.  The gate kernel of the unfused path sums with a shuffle tree, so
 * gates agree with engram_gate_add to fp32 rounding, not bit for bit; the
 * fused result itself is deterministic.  For at most 1536 tokens (decode
 * sizes, where the projection is only a wave or two of tiles) and for K below
 * 3200 (few k-blocks per tile, so the value tiles' wait and h traffic are not
 * hidden behind the main loop) the call runs engram_project and
 * engram_gate_add inside the workspace instead, which is faster there; the
 * results agree to the same rounding.
 *   e_d, wkv_packed_d, h_d, q_w_d, k_w_d   as engram_project (h_d updated in place)
 *   mask_d, eps, clamp, score_scale,
 *   gate_out_d                            as engram_gate_add
 *   workspace_d  device buffer of engram_project_gate_workspace_bytes(...)
 *                bytes, 256-byte aligned, owned by the caller; its contents
 *                on entry do not matter (the counters are zeroed on the stream)
 * A wait that runs out sets ENGRAM_ST_TIMEOUT in status_d. */
int engram_project_gate(const uint16_t* e_d, int64_t n_tokens, int64_t K, const uint16_t* wkv_packed_d,
                        int32_t hidden, int32_t hc, uint16_t* h_d, const float* q_w_d, const float* k_w_d,
                        const uint8_t* mask_d, float eps, float clamp, float score_scale, float* gate_out_d,
                        void* workspace_d, size_t workspace_bytes, int32_t* status_d, void* stream);

/* ------------------------------------------------------------------------ */
/* Projection + gate without device allocation                                */
/* ------------------------------------------------------------------------ */

/* Size of the library's static stage scratch (8 MiB). */
#define ENGRAM_STAGE_STATIC_SCRATCH_BYTES (8u << 20)

/* The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory where they run this stage, e.g. a
 * serving engine that has reserved all of HBM for its own pools and forbids
 * cudaMalloc on its hot path, or a plugin inside a host framework whose
 * allocator it does not own.
 *
 * Same result as engram_project followed by engram_gate_add on the same
 * arguments, but the two intermediates (partial sums and bf16 v) live in a
 * file-scope device array of ENGRAM_STAGE_STATIC_SCRATCH_BYTES, so the
 * caller passes only inputs and outputs and nothing is allocated.
 *   e_d, wkv_packed_d, q_w_d, k_w_d, mask_d (nullable): as engram_project /
 *   engram_gate_add; h_d: updated in place; gate_out_d: nullable.
 * Limit: round_up(engram_project_partials_bytes(n_tokens, hidden, hc), 256)
 *   + n_tokens * hidden * 2 must not exceed ENGRAM_STAGE_STATIC_SCRATCH_BYTES
 *   (about 728 tokens at hidden 5120, hc 4); larger requests return
 *   ENGRAM_E_RANGE with the limit in engram_last_error().
 * The array is part of the library image, so every GPU that loads the
 * library holds it until the process exits.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current, and a call looks it up again when the device's context is not the
 * one of the last lookup (after cudaDeviceReset); make the first call on a
 * device, and the first after a reset, before any stream capture.  All calls share
 * the array: calls that overlap on the GPU race on it.  Each call writes
 * every scratch element it reads, so no clearing is needed between calls. */
int engram_project_gate_add_noalloc(const uint16_t* e_d, int64_t n_tokens, int64_t K,
                                    const uint16_t* wkv_packed_d, int32_t hidden, int32_t hc,
                                    uint16_t* h_d, const float* q_w_d, const float* k_w_d,
                                    const uint8_t* mask_d, float eps, float clamp, float score_scale,
                                    float* gate_out_d, int32_t* status_d, void* stream);

/* ------------------------------------------------------------------------ */
/* Kernel selection                                                           */
/* ------------------------------------------------------------------------ */

/* Alternative kernels, for comparisons and profiling; the pages have no
 * counterpart.  The library picks its kernels by itself; these options
 * override that choice process-wide (every device and thread) from the next
 * call on.  All fields zero is the default choice.
 *   projection_cta  bf16 projection (engram_project, engram_project_gate):
 *                   0 single CTA up to 128 tokens and the CTA pair above,
 *                   1 the single-CTA kernel at every size, 2 the CTA pair at
 *                   every size
 *   gather_copy     row copies of the E4M3 + E8M0 gathers: 0 16-byte cp.async
 *                   copies, 1 one TMA bulk copy per row
 *   fp8_pair        block-FP8 projection: 0 single CTA, 1 CTA pair
 *   fp8_fused       engram_project_gate_fp8 above 1536 tokens: 0 projection
 *                   kernel then the gate kernel, 1 the fused kernel
 *   plain_launch    fused projection + gate kernels: 0 cooperative launch
 *                   (every CTA guaranteed resident), 1 plain launch, for
 *                   profilers that cannot replay a cooperative launch.  The
 *                   fused kernels' value tiles wait for gates that other CTAs
 *                   compute, so a plain launch is correct only while nothing
 *                   else runs on the GPU; otherwise such a wait may run out
 *                   and set ENGRAM_ST_TIMEOUT (no hang, no trap). */
typedef struct engram_kernel_options {
  int32_t projection_cta;
  int32_t gather_copy;
  int32_t fp8_pair;
  int32_t fp8_fused;
  int32_t plain_launch;
} engram_kernel_options;

/* Sets the options; ENGRAM_E_INVALID (nothing changed) for a null pointer or
 * a field out of range. */
int engram_set_kernel_options(const engram_kernel_options* opts);
/* Copies the options in force into *out. */
int engram_get_kernel_options(engram_kernel_options* out);

/* ------------------------------------------------------------------------ */
/* Test-data and diagnostics                                                  */
/* ------------------------------------------------------------------------ */

/* Fill a table with synthetic rows: row r holds the little-endian bytes of
 * SplitMix64 outputs number 33*r + j + 1 (j = 0..32) of a stream whose state
 * starts at `seed`; weight bytes equal to an E4M3 NaN code (0x7F, 0xFF) are
 * replaced by byte ^ 1 and each scale byte b becomes 120 + (b mod 11).  This
 * is input generation for tests and benchmarks, not part of the method.
 *   table_d  uint8 [n_rows][264], 8-byte aligned; device memory or a pinned
 *            (mapped) host buffer, which the kernel writes over NVLink-C2C */
int engram_fill_synthetic_table(uint8_t* table_d, int64_t n_rows, uint64_t seed, void* stream);

/* Fill a bf16-row table with synthetic rows: element c of row r is 16-bit
 * piece (c mod 4) of SplitMix64 output number r*(row_dim/4) + c/4 + 1 of the
 * stream at `seed`, with its 8 exponent bits replaced by 120 + (those bits
 * mod 11), so every value is finite with magnitude in [2^-7, 2^4).  Test and
 * benchmark input generation, not part of the method.
 *   table_d  bf16 [n_rows][row_dim], 8-byte aligned; row_dim a multiple of 4 */
int engram_fill_synthetic_rows_bf16(uint16_t* table_d, int64_t n_rows, int32_t row_dim, uint64_t seed,
                                    void* stream);

/* Diagnostic of the on-device modulo: out_d[i][j] = x_d[i] mod p_j + offset_j
 * for the layer's n_cols columns, computed by the same device routine as
 * engram_hash.  x_d: uint64 [n] (any 64-bit value); out_d: int64 [n][n_cols]. */
int engram_selftest_mod(const engram_layout* layout, int32_t layer, const uint64_t* x_d, int64_t n,
                        int64_t* out_d, void* stream);

/* Diagnostic of the bounded on-chip waits: one thread waits for something
 * that never happens, with the budget every kernel's waits use (2^31 SM
 * cycles, about a second), and the kernel then sets ENGRAM_ST_TIMEOUT in
 * status_d and returns -- no trap, no hang, the context stays usable.
 *   which      0: an mbarrier phase that no arrival completes (the TMA /
 *              tensor-core pipelines' waits); 1: a global counter that no
 *              CTA increments (the fused projection's wait for its block's
 *              gates)
 *   scratch_d  int32 [2] device scratch, zeroed by the call before the launch
 *   status_d   int32 status word (not cleared) */
int engram_selftest_wait(int32_t which, int32_t* scratch_d, int32_t* status_d, void* stream);

/* Thread-local message of the last failure (empty string if none). */
const char* engram_last_error(void);
/* Name of an ENGRAM_* return code. */
const char* engram_status_string(int code);
/* ENGRAM_ABI_VERSION of the loaded library. */
int engram_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_H */
