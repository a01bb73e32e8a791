// kernel_unit.cu -- one group of libspecverify's kernels, chosen by SPECV_UNIT
// at compile time, so that the groups compile in parallel:
//   1, 2   segment + row kernels, fp32 / bf16
//   3, 4   streaming kernel: greedy, and top-p (candidate groups and the
//          normaliser), fp32 / bf16
//   5, 6   streaming kernel: top-k candidate groups, fp32 / bf16
// Each group's unit defines its entries of kernel_table.h; the build links the
// units into one library.
#include "spec_kernels.cuh"
#include "kernel_table.h"

#ifndef SPECV_UNIT
#error "SPECV_UNIT selects the kernel group"
#endif

namespace specv_units {
namespace {
template <typename E, int MODE>
const void* stream_ptr() {
  return reinterpret_cast<const void*>(&spec_stream_kernel<E, MODE>);
}
}  // namespace

#if SPECV_UNIT == 1
const void* seg_f32(bool rag) {
  return rag ? reinterpret_cast<const void*>(&spec_seg_kernel<float, true>)
             : reinterpret_cast<const void*>(&spec_seg_kernel<float, false>);
}
const void* row_f32(bool rag) {
  return rag ? reinterpret_cast<const void*>(&spec_row_kernel<float, true>)
             : reinterpret_cast<const void*>(&spec_row_kernel<float, false>);
}
#elif SPECV_UNIT == 2
const void* seg_bf16(bool rag) {
  return rag ? reinterpret_cast<const void*>(&spec_seg_kernel<uint16_t, true>)
             : reinterpret_cast<const void*>(&spec_seg_kernel<uint16_t, false>);
}
const void* row_bf16(bool rag) {
  return rag ? reinterpret_cast<const void*>(&spec_row_kernel<uint16_t, true>)
             : reinterpret_cast<const void*>(&spec_row_kernel<uint16_t, false>);
}
#elif SPECV_UNIT == 3
const void* stream_f32_greedy() { return stream_ptr<float, kSMGreedy>(); }
const void* stream_f32_topp() { return stream_ptr<float, kSMTopP>(); }
#elif SPECV_UNIT == 4
const void* stream_bf16_greedy() { return stream_ptr<uint16_t, kSMGreedy>(); }
const void* stream_bf16_topp() { return stream_ptr<uint16_t, kSMTopP>(); }
#elif SPECV_UNIT == 5
const void* stream_f32_k() { return stream_ptr<float, kSMTopK>(); }
#elif SPECV_UNIT == 6
const void* stream_bf16_k() { return stream_ptr<uint16_t, kSMTopK>(); }
#endif

}  // namespace specv_units
