// Host-side interface between the C ABI (api.cu) and the kernel translation
// units (decode.cu, aux.cu).
#pragma once

#include <utility>

#include "common.cuh"

namespace da {

// Launches `kern` with programmatic stream serialisation (see grid_dep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct Choice {
  int engine;      // DA_ENGINE_CUDA_CORE or DA_ENGINE_MMA
  int variant;     // kVariantCore or kVariantMma (shared-memory layout)
  int rk;          // rows the kernel instance computes
  bool pingpong;   // CUDA cores, <= 4 rows: the two consumer warp groups take turns
  bool side_f8;    // FOLD far keys from an FP8 E4M3 side cache
  int stages;      // pipeline depth
  uint32_t smem;   // dynamic shared memory bytes
  int cluster;     // 0: flat partition; else CTAs per cluster of the cluster partition
};

// Picks the kernel instance for `rows` query rows per KV head (engine_hint:
// 0 automatic, 1 CUDA cores, 2 tensor cores) in `mode`; false when none
// exists or it does not fit in `max_smem` bytes of shared memory.
bool choose_kernel(int dtype, int d, int rows, int batch, int mode, int engine_hint, int stages,
                   int max_smem, bool side_f8, Choice* c);

cudaError_t prepare_decode(const Choice& c, int dtype, int d);

// Cluster partition (one cluster of CTAs per (sequence, KV head); decode
// kernels of decode_cluster.cu).  cluster_supported: whether an instance
// exists for the choice (shared-step engines, no FP8 side cache).
// prepare_cluster: sets the instance's attributes for clusters of up to
// `cluster` CTAs.  max_active_clusters: how many clusters of `cluster` CTAs
// the device holds at once (0 on error).
bool cluster_supported(const Choice& c, int dtype, int d);
// Sets c's cluster size and, with rank 0's receive slots for `cluster`
// partials in its layout, its pipeline depth (stages, or the deepest that
// fits when 0) and shared memory; false when nothing fits in max_smem.
bool fit_cluster(Choice* c, int dtype, int d, int batch, int cluster, int stages, int max_smem);
cudaError_t prepare_cluster(const Choice& c, int dtype, int d, int cluster);
int max_active_clusters(const Choice& c, int dtype, int d, int cluster);
cudaError_t launch_cluster(const Choice& c, int dtype, int d, const DecodeArgs& a,
                           const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& ms,
                           cudaStream_t st);

// The tcgen05 kernel (decode_tc.cu): attributes for the flat partition
// (cluster 0) or clusters of up to `cluster` CTAs, resident clusters, launch
// (the grid follows c.cluster).
cudaError_t tc_prepare(const Choice& c, int cluster);
int tc_max_active_clusters(const Choice& c, int cluster);
cudaError_t tc_launch(const Choice& c, const DecodeArgs& a, const CUtensorMap& mk,
                      const CUtensorMap& mv, const CUtensorMap& ms, cudaStream_t st);
cudaError_t launch_decode(const Choice& c, int dtype, int d, const DecodeArgs& a,
                          const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& ms,
                          cudaStream_t st);

struct AppendArgs {
  const void* k;
  const void* v;
  const int32_t* pos;
  const int32_t* block_table;
  void* k_cache;
  void* v_cache;
  void* k_side;
  uint32_t* status;
  int32_t B, n_new, H_kv, max_pages, num_pages;
  int32_t k_ring;   // rotated K of page P of sequence b at b * k_ring + ring_slot (0: paged)
  int32_t k_ring_sp;  // sink pages at the head of the ring
  int32_t side_f8;  // k_side holds E4M3 codes of k / side_scale
  float side_scale;
  float2 turn_freq[64];
};
cudaError_t launch_append(int dtype, int d, const AppendArgs& a, cudaStream_t st);

// Device, counter-region bytes and total workspace bytes of a plan; false for
// a null plan.
bool plan_workspace_layout(const da_plan_s* plan, int* device, size_t* counter_bytes,
                           size_t* workspace_bytes);

struct GatherOut {
  int32_t* positions;
  int64_t* phys_slot;
  int32_t* key_rope_pos;
  int32_t* q_rope_pos;
  int8_t* segment;
  int64_t capacity;
  int64_t* count;
};
cudaError_t launch_gather(const DecodeArgs& a, int b, int t, const GatherOut& o, cudaStream_t st);
cudaError_t launch_wait_timeout(uint32_t* status, cudaStream_t st);

}  // namespace da
