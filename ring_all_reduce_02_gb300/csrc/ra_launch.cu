// Dispatch to the (dtype, op) slices of ra_launch_op.cu, plus the
// op-independent kernels (all-gather and the ring's all-gather step).
#include "ra_ag.cuh"
#include "ra_bulk.cuh"
#include "ra_kernels.cuh"
#include "ra_order.cuh"
#include "ra_steps.cuh"

namespace ra {

#define RA_DECLARE_SLICE(DT, OP)                                                                  \
  cudaError_t launch_slice_##DT##_##OP(int kind, const Args& a, dim3 grid, cudaStream_t s);       \
  cudaError_t launch_ordered_slice_##DT##_##OP(bool is_rs, const OrderArgs& o, dim3 grid, cudaStream_t s); \
  cudaError_t launch_bulk_slice_##DT##_##OP(const BulkArgs& b, dim3 grid, size_t smem, cudaStream_t s); \
  cudaError_t configure_bulk_slice_##DT##_##OP(size_t smem); \
  cudaError_t launch_group_slice_##DT##_##OP(const GroupArgs& g, dim3 grid, cudaStream_t s);
#define RA_DECLARE_DT(DT) \
  RA_DECLARE_SLICE(DT, 0) RA_DECLARE_SLICE(DT, 1) RA_DECLARE_SLICE(DT, 2) RA_DECLARE_SLICE(DT, 3) RA_DECLARE_SLICE(DT, 4)
RA_DECLARE_DT(0)
RA_DECLARE_DT(1)
RA_DECLARE_DT(2)
RA_DECLARE_DT(3)

using SliceFn = cudaError_t (*)(int, const Args&, dim3, cudaStream_t);
using OrderedSliceFn = cudaError_t (*)(bool, const OrderArgs&, dim3, cudaStream_t);
#define RA_ROW(DT) {launch_slice_##DT##_0, launch_slice_##DT##_1, launch_slice_##DT##_2, launch_slice_##DT##_3, launch_slice_##DT##_4}
#define RA_OROW(DT)                                                                              \
  {launch_ordered_slice_##DT##_0, launch_ordered_slice_##DT##_1, launch_ordered_slice_##DT##_2, \
   launch_ordered_slice_##DT##_3, launch_ordered_slice_##DT##_4}
#define RA_BROW(DT)                                                                         \
  {launch_bulk_slice_##DT##_0, launch_bulk_slice_##DT##_1, launch_bulk_slice_##DT##_2, \
   launch_bulk_slice_##DT##_3, launch_bulk_slice_##DT##_4}
#define RA_CROW(DT)                                                                                   \
  {configure_bulk_slice_##DT##_0, configure_bulk_slice_##DT##_1, configure_bulk_slice_##DT##_2, \
   configure_bulk_slice_##DT##_3, configure_bulk_slice_##DT##_4}
using BulkSliceFn = cudaError_t (*)(const BulkArgs&, dim3, size_t, cudaStream_t);
using BulkConfigureFn = cudaError_t (*)(size_t);
#define RA_GROW(DT)                                                                            \
  {launch_group_slice_##DT##_0, launch_group_slice_##DT##_1, launch_group_slice_##DT##_2, \
   launch_group_slice_##DT##_3, launch_group_slice_##DT##_4}
using GroupSliceFn = cudaError_t (*)(const GroupArgs&, dim3, cudaStream_t);
const SliceFn kSlices[4][5] = {RA_ROW(0), RA_ROW(1), RA_ROW(2), RA_ROW(3)};
const OrderedSliceFn kOrderedSlices[4][5] = {RA_OROW(0), RA_OROW(1), RA_OROW(2), RA_OROW(3)};
const BulkSliceFn kBulkSlices[4][5] = {RA_BROW(0), RA_BROW(1), RA_BROW(2), RA_BROW(3)};
const BulkConfigureFn kBulkConfigure[4][5] = {RA_CROW(0), RA_CROW(1), RA_CROW(2), RA_CROW(3)};
const GroupSliceFn kGroupSlices[4][5] = {RA_GROW(0), RA_GROW(1), RA_GROW(2), RA_GROW(3)};

template <int DT, int kUnroll>
cudaError_t launch_ag_tile(const Args& a, dim3 grid, cudaStream_t s) {
  constexpr uint32_t smem = ag_tile_bytes<kUnroll>();
  if constexpr (smem > 48 * 1024) {  // above the default limit of dynamic shared memory
    const cudaError_t err =
        cudaFuncSetAttribute(ag_tile_kernel<DT, kUnroll>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  return launch_programmatic(ag_tile_kernel<DT, kUnroll>, grid, kAgThreads, smem, s, a);
}

template <int DT>
cudaError_t launch_op_free(int kind, const Args& a, dim3 grid, cudaStream_t s) {
  if (kind == KIND_ALLGATHER && a.shape == kShapeAgBase + AG_TILE) {
    switch (ag_plan_for(a.nranks).unroll) {
      case 1: return launch_ag_tile<DT, 1>(a, grid, s);
      case 2: return launch_ag_tile<DT, 2>(a, grid, s);
      default: return launch_ag_tile<DT, 4>(a, grid, s);
    }
  }
  if (kind == KIND_RING_AG_STEP) return launch_ring_ag_step<DT>(a, grid, s);
  return launch_programmatic(ag_copy_kernel<DT, AgShape>, grid, AgShape::kThreads, 0, s, a);
}

cudaError_t launch_kernel(int kind, int dtype, int op, const Args& a, dim3 grid, cudaStream_t s) {
  if (dtype < 0 || dtype > 3 || op < 0 || op > 4) return cudaErrorInvalidValue;
  if (kind == KIND_ALLGATHER || kind == KIND_RING_AG_STEP) {
    switch (dtype) {
      case DT_F32: return launch_op_free<DT_F32>(kind, a, grid, s);
      case DT_F16: return launch_op_free<DT_F16>(kind, a, grid, s);
      case DT_BF16: return launch_op_free<DT_BF16>(kind, a, grid, s);
      default: return launch_op_free<DT_I32>(kind, a, grid, s);
    }
  }
  return kSlices[dtype][op](kind, a, grid, s);
}

cudaError_t launch_ordered_kernel(bool is_rs, int dtype, int op, const OrderArgs& o, dim3 grid, cudaStream_t s) {
  if (dtype < 0 || dtype > 3 || op < 0 || op > 4) return cudaErrorInvalidValue;
  return kOrderedSlices[dtype][op](is_rs, o, grid, s);
}

cudaError_t launch_group_kernel(int dtype, int op, const GroupArgs& g, dim3 grid, cudaStream_t s) {
  if (dtype < 0 || dtype > 3 || op < 0 || op > 4) return cudaErrorInvalidValue;
  return kGroupSlices[dtype][op](g, grid, s);
}

cudaError_t configure_bulk_kernel(int dtype, int op, size_t smem) {
  if (dtype < 0 || dtype > 3 || op < 0 || op > 4) return cudaErrorInvalidValue;
  return kBulkConfigure[dtype][op](smem);
}

cudaError_t launch_bulk_kernel(int dtype, int op, const BulkArgs& b, dim3 grid, size_t smem, cudaStream_t s) {
  if (dtype < 0 || dtype > 3 || op < 0 || op > 4) return cudaErrorInvalidValue;
  return kBulkSlices[dtype][op](b, grid, smem, s);
}

}  // namespace ra
