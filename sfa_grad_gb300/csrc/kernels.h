// Internal launcher declarations shared by the C-ABI host code and the kernels.
#pragma once
#include "common.cuh"

namespace sfa {

constexpr int kModeBwd = 0;       // S and dP -> P, dS
// S -> partial max / sum statistics; the per-token kernel (sdp.cu) also
// stages P relative to each partial max (one partial per 32 keys)
constexpr int kModeFwdStats = 1;

// Score / softmax-gradient kernel (sdp.cu).  The staged P^T / dS^T rows go
// through the store maps maps.Pw / maps.dSw.
template <typename T>
cudaError_t launch_sdp(const Maps& maps, const Prob& p, int mode, float* tile_stats, int* gerr, int nsm,
                       cudaStream_t st);

// Key-major dK / dV for block-sparse indices (kvb.cu): group the chunk's
// (token, index) pairs by block start (count, scan, scatter), then accumulate
// every group's block in tensor memory and add it to acc once.  res >= 0
// (deterministic mode; entries sorted within each group): only the groups
// whose start is res modulo bs, whose blocks share no key row.
// pst / dsst (optional): the staged P^T / dS^T; the rows no group covers
// (pairs left out, padding slots) are zeroed.  tile_stats (optional, the
// forward's per-pair statistics): a left-out pair's entries are set to
// {-inf, 0}.
cudaError_t launch_blk_count(const Prob& p, int* cnt, void* pst, void* dsst, float* tile_stats, cudaStream_t st);
// nres (optional, bs entries): non-empty bins per residue modulo bs.
cudaError_t launch_blk_scan(const int* cnt, int nbins, int* cursor, int* groups, int* gbeg, int* ngroups, int bs,
                            int* nres, cudaStream_t st);
cudaError_t launch_blk_scatter(const Prob& p, int* cursor, int* entries, cudaStream_t st);
template <typename T>
cudaError_t launch_kvb(const BlkMaps& maps, const Prob& p, int bs, const int* groups, const int* gbeg,
                       const int* ngroups, const int* entries, float* acc, int res, const int* nres, int* gerr,
                       int nsm, cudaStream_t st);

// Key-major scores for block-sparse indices (sdpb.cu): per group of pairs
// sharing a block start, S (and dP) of packs of 128 / GK tokens against the
// block's resident key (and value) rows.  mode kModeBwd writes the pairs'
// staged P^T / dS^T rows; kModeFwdStats the pairs' partial statistics
// (tile_stats, (token, index, head) x {max, sum}) and their P^T rows relative
// to each pair's max.
template <typename T>
cudaError_t launch_sdpb(const Maps& maps, const Prob& p, int mode, const int* groups, const int* gbeg,
                        const int* ngroups, const int* entries, void* pst, void* dsst, float* tile_stats, int* gerr,
                        int nsm, cudaStream_t st);

// Key-side and query-side contractions in one launch, two pipelines per CTA
// (kvq.cu): key-side reductions into acc, dQ / dQRope out.  tile_group: key
// tiles per key-side work item, at least 1 (items run tile-group major; a
// group of all tiles gives token-major order).  part:
// deterministic mode; acc is then the chunk's partial-row buffer (bf16
// elements) and every valid (token, slot) row is stored there instead of
// reduced.
template <typename T>
cudaError_t launch_kvq(const Maps& maps, const Prob& p, float* acc, void* dq, void* dqr, int tile_group, bool part,
                       int* gerr, int nsm, cudaStream_t st);

// dQ / dQRope for block-sparse indices with at most 64 heads (dqb.cu):
// features on the MMA's M, heads on N, over each token's selected blocks.
// pv: the companion forward's O = P V instead (value rows; dq is the
// output, dqr unused), from P staged by sdpb's statistics pass relative to
// each (token, block) pair's max and rescaled to the final statistics
// p.smax, p.ssum; part_stats: that pass's (pair, head) x {max, sum}.
template <typename T>
cudaError_t launch_dqb(const Maps& maps, const Prob& p, bool pv, void* dq, void* dqr, const float* part_stats,
                       int* gerr, int nsm, cudaStream_t st);

// Companion forward's output O = P V over each token's selected keys (dq.cu),
// from the P staged by sdp.cu's statistics pass relative to each 32-key
// group's max, rescaled per (group, head) to the final statistics p.smax,
// p.ssum.  part_stats: that pass's (token, Kpad / 32 groups, head) x {max of
// the raw score, sum}.
template <typename T>
cudaError_t launch_pv(const Maps& maps, const Prob& p, const float* part_stats, void* out, int* gerr, int nsm,
                      cudaStream_t st);

// Small kernels (prep.cu).
cudaError_t launch_rowtab(const Prob& p, cudaStream_t st);
cudaError_t launch_batch_prefix(const Prob& p, int B, const int* act_q, const int* act_kv, int* batch_ofs, int* gerr,
                                cudaStream_t st);
cudaError_t launch_meta(const Prob& p, int layout, int B, int S1, int S2, int mode, const int* act_q, const int* act_kv,
                        int* batch_ofs, TokMeta* meta, int* gerr, cudaStream_t st);
// Dsum of tokens tok0 .. tok0 + ntok - 1 (all heads).
template <typename T>
cudaError_t launch_dsum(const Prob& p, int tok0, int ntok, float* dsum, cudaStream_t st);
template <typename T>
cudaError_t launch_cast(const float* acc, int T2, void* dk, void* dkr, void* dv, int has_rope, cudaStream_t st);
// ntiles: partial statistics per token (32-key groups, or block indices).
cudaError_t launch_stats_combine(const Prob& p, const float* tile_stats, int ntiles, float* smax, float* ssum,
                                 cudaStream_t st);

// Records a message for sfa_last_error_message on the calling thread (api.cu).
void set_last_error(const char* msg);

// Deterministic key-side reduction (det.cu): counting sort of the chunk's
// (kv row, token, slot) entries by row (count, then launch_blk_scan over the
// T2 rows, scatter, per-row sort), then one fixed-order sum per row.
cudaError_t launch_det_count(const Prob& p, int* cnt, cudaStream_t st);
cudaError_t launch_det_scatter(const Prob& p, int* cursor, int* ent, cudaStream_t st);
// Sorts each row's segment of entry ids ascending: long_segs = false sorts the
// segments of up to 1024 entries, true the longer ones (two launches).
cudaError_t launch_det_sort(const Prob& p, const int* gbeg, const int* ngroups, int* ent, int* scratch, bool long_segs,
                            cudaStream_t st);
cudaError_t launch_det_reduce(const Prob& p, const int* groups, const int* gbeg, const int* ngroups, const int* ent,
                              const uint16_t* partials, float* acc, cudaStream_t st);

}  // namespace sfa
