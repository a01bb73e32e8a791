// kernel_table.h -- the kernel groups of libspecverify, one per compilation of
// kernel_unit.cu, so that they compile in parallel.  Each returns the address
// of a kernel for the host's launch calls.
#pragma once

namespace specv_units {

// segment + row kernels (the two-kernel path); rag: a ragged call
const void* seg_f32(bool rag);
const void* row_f32(bool rag);
const void* seg_bf16(bool rag);
const void* row_bf16(bool rag);
// the one-launch streaming kernel: greedy; top-p; top-k candidate groups
const void* stream_f32_greedy();
const void* stream_bf16_greedy();
const void* stream_f32_topp();
const void* stream_bf16_topp();
const void* stream_f32_k();
const void* stream_bf16_k();

}  // namespace specv_units
