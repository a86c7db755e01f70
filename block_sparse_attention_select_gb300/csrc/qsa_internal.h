// Shared host/device definitions of the QSA library (not part of the ABI).
#pragma once
#include <cstddef>
#include <cstdint>

namespace qsa {

// Device status bits (the host maps the highest-priority one to qsa_status).
enum : uint32_t {
    ST_BAD_PAGE = 1u << 0,
    ST_BAD_ROW = 1u << 1,       // row_req out of range or row longer than allowed
    ST_TIMEOUT = 1u << 2,
};

constexpr int TILE_M = 128;      // positions per scorer tile (MMA M, TMEM lanes)
constexpr int HEAD_DIM = 128;    // index-key dimension (MMA K per head)
constexpr int N_MAX = 256;       // MMA N: (query rows of a group) x heads
constexpr int KSTAGES = 4;       // key tiles in flight per CTA
constexpr int EPI_WARPS = 16;    // 4 per TMEM lane quarter, each owning 64 accumulator columns
constexpr int SCORE_THREADS = 64 + 32 * EPI_WARPS;   // warp 0 TMA, warp 1 MMA, then epilogue

// Candidate lists of the filter pass.  Key tile t of row r has four quarters
// q of 32 positions (t*128 + q*32 + i, i < 32):
//   cand_mask[r*tiles_ld*4 + 4t + q], bit i: position t*128 + q*32 + i passed;
//   the j-th passing position of quarter q (ascending i) has its score at
//   cand_score[(t*R + r)*128 + 4j + q].
// Each (tile, row) owns one 512-byte region whose "slot row" j holds the j-th
// candidate of each of the four quarters, so the few candidates of a tile
// (the filter keeps a few percent of the positions) share the region's first
// sectors and the four quarter warps of a tile fill those sectors together.
// Rows of one tile are 512 bytes apart, a compile-time stride: the scorer
// addresses a row's slot with an immediate offset.  The region is as large as
// the dense logits of the same rows, which it replaces on the filter path (a
// row the selector re-scores reuses it).  tiles_ld is a multiple of 8, which
// keeps each row's mask words in 128-byte lines of their own.
constexpr int TH_STAGE = 16384;  // sampled scores of one row the threshold kernel holds in shared memory

// A group: consecutive query rows of one request that share every key tile.
struct Group {
    int32_t row0;      // first query row
    int32_t nrows;     // rows in the group (<= N_MAX / H)
    int32_t req;       // request index (row of the block table)
    int32_t vmax;      // longest visible length in the group (positions)
    int32_t vmin;      // shortest visible length in the group
};

// Plan written by the plan kernel into the workspace.
struct Plan {
    int32_t n_groups;
    int32_t n_items;           // (group, tile) items over all groups
    int32_t n_sample_items;    // items of the sampled tiles only
    int32_t any_fallback;      // set by the candidate selector
};

enum ScoreMode : int32_t {
    SCORE_LOGITS = 0,      // logits for j < V_r (and -inf up to the tile end when pad_inf)
    SCORE_SAMPLE = 1,      // sampled tiles only, into the sample matrix
    SCORE_FILTER = 2,      // append (score, j) with score >= tau_r to the candidate lists
    SCORE_BLOCKMAX = 3,    // block scorer (its own kernel): per (row, head) the max over each 128-token block
};

struct ScoreParams {
    const float *w;             // [R, H]
    const int32_t *row_vis;     // sanitised V_r [R]
    const Group *groups;
    const int32_t *item_prefix;     // [n_groups + 1] items before group g
    const int32_t *sample_prefix;   // [n_groups + 1]
    const Plan *plan;
    const int32_t *block_table;
    int32_t max_pages;
    int32_t num_pages;
    int32_t page_pos;           // positions per page
    int32_t page_box;           // rows per TMA box = min(page_pos, TILE_M)
    int32_t page_pos_shift;     // log2(page_pos), log2(page_box), log2(sample_stride): all
    int32_t page_box_shift;     // three are powers of two, and divisions by runtime values
    int32_t sample_shift;       // cost ~20 instructions on the producer's critical path
    int32_t H;
    int32_t R;
    int32_t mode;
    int32_t sample_stride;      // tiles between sampled tiles
    // outputs
    float *out;                 // logits [R, ld] or sample matrix [R, ld]
    int64_t ld;
    int32_t pad_inf;            // LOGITS: write -inf for V_r <= j < tile end (j < ld)
    const float *tau;           // FILTER: per-row threshold
    float *cand_score;          // FILTER: [tiles_ld, R, 128] candidate scores (layout above)
    uint32_t *cand_mask;        // FILTER: [R, tiles_ld * 4] passing positions of each quarter
    int32_t tiles_ld;           // key tiles per row in the candidate arrays (multiple of 8)
    uint32_t *status;
    uint64_t wait_limit_ns;
    // BLOCKMAX (the M3-style block scorer, score_blockrows_kernel): rows are
    // virtual rows v = h * blk_rows + r, one per (query row r, KV head h); a
    // group's req is the virtual request h * blk_reqs + b.  Queries are read
    // through a 3-D map [rows][H][128] and keys through [tokens][H][128], two
    // 128-token pages per tile.
    int32_t blk_heads;          // KV heads (0 outside BLOCKMAX)
    int32_t blk_reqs;           // requests of the block table
    int32_t blk_rows;           // query rows
};

enum SelectMode : int32_t {
    SEL_DENSE = 0,      // row r = logits[r, 0:V_r]
    SEL_THRESH = 2,     // row r = sample row; writes tau_r
    SEL_CAND = 3,       // row r = candidate list; flags the row when it cannot be trusted
};

struct SelectParams {
    int32_t mode;
    int32_t R;
    int32_t k;
    const float *logits;        // DENSE: logits; THRESH: sample matrix
    int64_t ld;
    int64_t max_len;            // largest valid V_r (longer rows are clamped and flagged)
    const int32_t *row_vis;     // V_r
    const float *cand_score;    // CAND: lists written by the filter scorer
    const uint32_t *cand_mask;
    int32_t tiles_ld;
    int32_t cap;                // THRESH: rows up to this length keep every position; CAND: list capacity
    int32_t *row_flag;          // CAND: 1 for rows that took the in-kernel fallback, else 0
    Plan *plan;
    // CAND fallback: a row whose list cannot be trusted is re-scored (plain
    // FP32 arithmetic) into its own regions of the candidate array (fb_scores
    // = cand_score, position j of row r at ((j / 128) * R + r) * 128 + j % 128)
    // and selected densely
    const uint16_t *q;          // FP16 bits [R, H, 128]
    const float *w;             // [R, H]
    const uint16_t *k_cache;    // FP16 bits [num_pages, page_pos, 128]
    const int32_t *block_table;
    const int32_t *row_req;
    int32_t H, max_pages, num_pages, page_pos;
    float *fb_scores;
    // THRESH
    int32_t sample_stride;
    float *tau;
    float oversample;           // expected candidates / k
    // outputs
    int32_t *out_idx;
    float *out_val;
    int32_t smem_cap;           // elements the CTA can hold in shared memory
    uint32_t *status;
    // DENSE: with out_heads > 1 the R = out_heads * n rows are virtual rows
    // v = h * n + r and row v's output goes to row r * out_heads + h
    int32_t out_heads;
};

// Index-key producer (the step before the indexer): see qsa_produce.cu.
struct ProduceParams {
    const void *x;              // FP16 [T, 128] token keys, request after request
    const float *pool_logit;    // [T] or nullptr (equal weights)
    const int32_t *seq_start;   // [n_reqs + 1] row offsets into x
    const int32_t *pos_start;   // [n_reqs] position of each request's first new token
    const float *norm_weight;   // [128], 16-byte aligned
    const float *rope_table;    // [rope_blocks, rope_dim], 16-byte aligned
    void *k_cache;              // FP16 [num_pages, page_positions, 128]
    const int32_t *block_table; // [>= n_reqs, max_pages]
    int32_t n_reqs, num_pages, page_positions, page_shift, max_pages;
    int32_t rope_dim, rope_blocks, window;
    float eps;
    uint32_t *status;
};

// Sparse-attention consumer (the step after the indexer): see qsa_attend.cu.
struct AttendParams {
    const void *q;              // FP16 [rows, hq, 256]
    const void *k_cache;        // FP16 [num_pages, page_tokens, hkv, 256]
    const void *v_cache;        // same layout
    const int32_t *block_table; // [num_reqs, max_pages]
    const int32_t *row_req;     // [rows]
    const int32_t *row_token;   // [rows]
    const int32_t *sel;         // [rows, k] selected index positions, -1 = none
    float *out;                 // FP32 [rows, hq, 256]
    int32_t rows, hq, hkv, k, num_pages, page_tokens, page_shift, num_reqs, max_pages;
    float scale;
    uint32_t *status;
    uint64_t wait_limit_ns;     // a tensor-core wait that takes longer gives up (QSA_ERR_TIMEOUT)
};

// Launchers (one translation unit each); return cudaError_t as int.  With
// `overlap` the launch carries programmatic stream serialization: the kernel
// may be scheduled while the previous kernel of the stream is still running
// (once every CTA of that kernel has allowed it) and waits for that kernel's
// completion itself before it touches global memory.  The first kernel of a
// call is launched without it, so a call never overlaps the caller's work.
// tile_shift: log2 of the key positions per work item (7: the scorers'
// 128-position tiles; 8: the block scorer's 256-token tiles)
int launch_plan(const int32_t *row_req, const int32_t *row_visible, int32_t R, int32_t group_rows,
                int32_t num_reqs, int64_t max_len, int32_t sample_stride, int32_t *row_vis,
                Group *groups, int32_t *item_prefix, int32_t *sample_prefix, Plan *plan,
                uint32_t *status, void *stream, int32_t tile_shift = 7);
int launch_score(const ScoreParams &p, const void *tmap_q, const void *tmap_k, const void *tmap_k128,
                 int grid, bool overlap, void *stream);
// Block scorer with the virtual rows on the TMEM lanes (BLOCKMAX): groups of
// up to BR_ROWS rows of one head (two MMA halves of 128 rows), tiles of 2
// blocks (256 tokens); tmap_q3 is the query map [rows][H][128] with boxes
// 64 x 1 x BR_ROWS, tmap_k the key map [tokens][H][128] with boxes 64 x 1 x 128
// (one page).
constexpr int BR_ROWS = 256;
int launch_score_blockrows(const ScoreParams &p, const void *tmap_q3, const void *tmap_k, int grid, bool overlap,
                           void *stream);
// cluster_pref (SEL_CAND only): CTAs per row of the candidate selector, 0 =
// automatic (a thread-block cluster per row when rows are fewer than SMs, its
// size from the device's occupancy query), 1 = one CTA per row, 2 / 4 / 8 =
// that cluster size (capped by the query)
int launch_select(const SelectParams &p, int grid, bool overlap, void *stream, int cluster_pref = 0);
size_t select_smem_bytes(int32_t smem_cap);
// cand_kernel's shared memory; fb_cap (if given): keys its fallback stages
size_t cand_smem_bytes(int32_t k, int32_t cap, bool pos16, int32_t *fb_cap = nullptr);
size_t cand_cluster_smem_bytes(int32_t k, int32_t cap);
extern int last_cluster;    // CTAs per row of the most recent candidate-selector launch
uint32_t score_smem_bytes();
int launch_pad(float *logits, int64_t ld, int32_t R, const int32_t *row_vis, bool overlap, void *stream);
// Block scorer rows: for v = h * R + r, vreq[v] = row_req[r] + h * num_reqs (or
// -1 when row_req[r] is out of range), vtok[v] = row_token[r] + 1 visible
// tokens (0 and flagged when negative), vblk[v] = visible 128-token blocks.
int launch_block_rows(const int32_t *row_req, const int32_t *row_token, int32_t R, int32_t H,
                      int32_t num_reqs, int32_t *vreq, int32_t *vtok, int32_t *vblk, uint32_t *status,
                      void *stream);
int launch_produce(const ProduceParams &p, int32_t max_tokens, void *stream);
int launch_rope_table(float *table, int32_t n_blocks, int32_t rope_dim, double theta, void *stream);
int launch_attend(const AttendParams &p, void *stream);

}  // namespace qsa
