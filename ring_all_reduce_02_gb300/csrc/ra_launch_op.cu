// One (dtype, op) slice of the kernel instantiations. The build compiles this
// file once per pair, with RA_SLICE_DT and RA_SLICE_OP set, so the twenty
// slices compile in parallel; ra_launch.cu dispatches to them.
#include "ra_bulk.cuh"
#include "ra_kernels.cuh"
#include "ra_order.cuh"
#include "ra_steps.cuh"

#if !defined(RA_SLICE_DT) || !defined(RA_SLICE_OP)
#error "compile with -DRA_SLICE_DT=<dtype id> -DRA_SLICE_OP=<op id>"
#endif

#define RA_CAT3_(a, b, c) a##_##b##_##c
#define RA_CAT3(a, b, c) RA_CAT3_(a, b, c)

namespace ra {
cudaError_t RA_CAT3(launch_slice, RA_SLICE_DT, RA_SLICE_OP)(int kind, const Args& a, dim3 grid, cudaStream_t s) {
  if (kind == KIND_RING_RS_STEP) return launch_ring_rs_step<RA_SLICE_DT, RA_SLICE_OP>(a, grid, s);
  return launch_op<RA_SLICE_DT, RA_SLICE_OP>(kind, a, grid, s);
}
cudaError_t RA_CAT3(launch_ordered_slice, RA_SLICE_DT, RA_SLICE_OP)(bool is_rs, const OrderArgs& o, dim3 grid,
                                                                    cudaStream_t s) {
  return launch_ordered_op<RA_SLICE_DT, RA_SLICE_OP>(is_rs, o, grid, s);
}
cudaError_t RA_CAT3(launch_bulk_slice, RA_SLICE_DT, RA_SLICE_OP)(const BulkArgs& b, dim3 grid, size_t smem,
                                                                 cudaStream_t s) {
  return launch_bulk_op<RA_SLICE_DT, RA_SLICE_OP>(b, grid, smem, s);
}
cudaError_t RA_CAT3(configure_bulk_slice, RA_SLICE_DT, RA_SLICE_OP)(size_t smem) {
  return configure_bulk_op<RA_SLICE_DT, RA_SLICE_OP>(smem);
}
cudaError_t RA_CAT3(launch_group_slice, RA_SLICE_DT, RA_SLICE_OP)(const GroupArgs& g, dim3 grid, cudaStream_t s) {
  return launch_group_op<RA_SLICE_DT, RA_SLICE_OP>(g, grid, s);
}
}  // namespace ra
