// Internal interface between the C-ABI layer and the beam-step kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vbs {

constexpr int WMAX = 16;          // beams per sentence
constexpr int KMAX = 2 * WMAX;    // candidates kept per row (2W)
constexpr int PART_KEYS = 256;    // keys one row merge can hold (partials x K)
constexpr int CAND_CAP = 288;     // candidate buffer per warp: K + one 32-lane x 8-element vector

// Paged KV cache: one sentence's blocks live in [b*S, (b+1)*S) of the pool.
struct PagedArgs {
  int B, W, S, MB, block, L, H;
  int64_t block_bytes;            // bytes of one pool block
  int64_t slot_bytes;             // bytes of one position within one (l, kv, h) run
  char* pool;
  int32_t* table;                 // [R, MB]
  int32_t* nblk;                  // [R]
  int32_t* refcnt;                // [B*S]
  int32_t* stack;                 // [B*S]
  int32_t* top;                   // [B]
  int4* tasks;                    // [R]: sentence b's tasks in [b*W, (b+1)*W) (src block, dst block, filled slots, -)
  int task_cap;                   // R
  unsigned long long* cow_slots;  // filled slots copied, summed (x L*2*H runs)
  int* status;
};

struct BsArgs {
  const void* logits;
  int64_t ld;
  int dtype;
  int B, W, V, K, R;
  int64_t per;                    // elements of the flattened [R, V] space per CTA
  int P;                          // partial slots per row
  float* scores;
  int32_t* seqs;
  int seq_ld;                     // max_len + 1
  int32_t* beam_idx;
  int32_t* tokens;
  int32_t* all_done_out;          // optional, caller's
  int32_t* all_done_dev;          // the context's own flag
  int t;                          // 1-based step number (finalize: steps run)
  int eos, bos, pad, early_stopping, lp_kind, max_len;
  double alpha;
  double lp_t;                    // lp(t): normalises an EOS hit of this step (finalize: lp(steps run))
  double lp_bound;                // lp of the stopping test's best attainable length
  float lp_tf, lp_boundf;         // the same two in fp32 (the walk and the stopping test run in fp32)
  // workspace
  float* part_M;
  float* part_l;
  unsigned long long* part_key;
  unsigned* rtopk_bar;            // [R] the two-pass ablation's per-row bar (ordered logit bits)
  int* row_one;                   // [R] all 1: the two-pass ablation writes one partial slot per row
  int vbase;                      // token id of the first logit column (a vocabulary shard's offset)
  // vocabulary shards: up to shard_max partials per row, merged by the merge kernel
  int shard_max;
  float* shard_M;                 // [R][shard_max]
  float* shard_l;
  unsigned long long* shard_key;  // [R][shard_max][K]
  int* row_ns;                    // [R] the number of shards of the current merge
  int* row_p0;                    // [R] the first CTA whose range holds row r
  int* row_np;                    // [R] the number of CTAs (partials) holding row r
  int* done_count;                // sentences finished (step-local counter)
  int cluster;                    // 0: flat split + merge kernel; C: a cluster of C CTAs per sentence
  int* done;
  // finished sets
  double* fin_ns;
  int* fin_len;
  int* fin_serial;
  int32_t* fin_tok;
  int* fin_count;
  int* fin_next;
  double* fin_worst;
  int* status;
  // cluster mode: the paged KV remap of the step, fused after the sentence merge (kv_fuse != 0)
  int kv_fuse;
  int kv_t;                       // t_valid of the remap
  PagedArgs kv;
};

int launch_bs_step(const BsArgs& a, int grid, bool vector_ok, cudaStream_t s);
bool bs_can_fuse_remap(const BsArgs& a, const PagedArgs& kv);
int launch_bs_step_two_pass(const BsArgs& a, bool vector_ok, cudaStream_t s);
// one vocabulary shard's per-row partial (max, scaled sum, K best keys) into a caller buffer laid
// out as shard_partial_layout gives, and the merge of n such buffers
void shard_partial_layout(int R, int K, size_t* off_l, size_t* off_key, size_t* bytes);
int launch_bs_shard_partial(const BsArgs& a, bool vector_ok, void* partial, cudaStream_t s);
int launch_bs_merge_shards(const BsArgs& a, int n_shards, const void* partials, cudaStream_t s);
int launch_bs_reset(const BsArgs& a, cudaStream_t s);
int launch_bs_finalize(const BsArgs& a, const float* scores, const int32_t* seqs, int n_ret, int32_t* out_seqs,
                       int32_t* out_len, float* out_score, cudaStream_t s);
constexpr int BS_NSLOT = 4;       // row segments one stream CTA holds (cluster mode: W / C <= this)
int bs_threads_per_cta();
int bs_ctas_per_sm();

// bs_expand_static: scratch in a static device array of this size; rows at most.  With
// R >= the CTA count every row has P = 2 partial slots, so the carve is at most
// R * (2 * (8 + 8 K) + 8) + 4 B bytes plus alignment: 4,392,960 at R = 8192, W = 16 (K = 32).
constexpr size_t STATIC_SCRATCH_BYTES = size_t{9} << 19;   // 4.5 MiB
constexpr int STATIC_MAX_ROWS = 8192;
int launch_bs_expand_static(BsArgs a, int grid, bool vector_ok, float* scores_out, cudaStream_t s);

// KV reorder
struct KvGeom {
  int L, H, rows;
  int64_t seg_stride;             // bytes between consecutive (l, kv, r, h) segments
  int64_t copy_bytes;             // bytes copied per segment
};
int launch_kv_naive(const KvGeom& g, const void* src, void* dst, const int32_t* beam_idx, bool bulk_ok,
                    int elem_bytes, int* status, int num_sms, cudaStream_t s);

int launch_kv_paged_remap(const PagedArgs& a, const int32_t* beam_idx, int t_valid, cudaStream_t s);
int launch_kv_paged_cow(const PagedArgs& a, bool bulk_ok, int num_sms, cudaStream_t s);

// blockwise parallel decoding; mode VBS_BPD_EXACT / _TOPK / _DISTANCE with its parameter,
// and the minimum accepted block (1 = none)
struct BpdCrit {
  int mode, param, min_accept;
};
int launch_bpd_propose(const void* logits, int B, int k, int V, int dtype, bool vec_ok, int32_t* proposals,
                       cudaStream_t s);
int launch_bpd_verify(const void* logits, const int32_t* proposals, int B, int k, int V, int dtype, bool vec_ok,
                      int eos, const BpdCrit& crit, int32_t* khat, int32_t* next, int* status, int num_sms,
                      cudaStream_t s);

// in-run memory peaks (measurement): a vector copy, and a read-only stream (mode 0: vector
// loads, mode 1: a bulk-copy ring into shared memory)
int launch_peak_copy(const void* src, void* dst, int64_t bytes, int grid, cudaStream_t s);
int launch_peak_read(const void* src, int64_t bytes, int grid, int mode, uint32_t* sink, int* status, cudaStream_t s);

// the first failed device bounds check of each file in the checked build (0: none)
unsigned long long bs_check_record();
unsigned long long kv_check_record();
unsigned long long bpd_check_record();

}  // namespace vbs
