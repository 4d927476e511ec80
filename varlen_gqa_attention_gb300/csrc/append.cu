// append.cu - the step's keys and values written into the column store before attention.
//
// "[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV columns", #24074
// commit message in its stack: each update-and-attend becomes an in-graph write to slot
// (position % rows) * columns + seq_cols[i], then the attention over the column store.
// Here packed row q_start + i of a live segment (valid, not overlapping: the scheduler's
// verdict, so the append and the attention agree on which segments exist) holds position
// p = kv_end - q_len + i and is copied, every KV head, to store row p % rows of the
// segment's column; rows with p < 0 write nothing.  The kernel runs between the scheduler
// and the attention kernels of one call, so the attention reads what it wrote.
#include "common.cuh"

namespace sdpa {

// One CTA row per segment (blockIdx.x), gridDim.y CTAs sharing its rows; 16-byte copies.
__global__ void __launch_bounds__(kAppendThreads) sdpa_append_kernel(AppendArgs A) {
  griddep_wait();  // the scheduler's segment records
  griddep_launch();
  const SegRec sg = A.segs[blockIdx.x];
  if (sg.route == kRouteNone || sg.q_len <= 0) return;
  const int chunks = A.Hkv * (A.D / 8);  // 16-byte chunks of one packed row
  const int64_t n = (int64_t)sg.q_len * chunks;
  const int64_t base = (int64_t)sg.kv_end - sg.q_len;  // position of row 0
  for (int64_t idx = (int64_t)blockIdx.y * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.y * blockDim.x) {
    const int64_t i = idx / chunks;
    const int rem = (int)(idx - i * chunks);
    const int h = rem / (A.D / 8), c = rem % (A.D / 8);
    const int64_t p = base + i;
    if (p < 0) continue;
    const int64_t src = ((int64_t)sg.q_start + i) * A.new_rs + (int64_t)h * A.new_hs + c * 8;
    const int64_t dst = (((p % A.rows) * A.cols + sg.col) * A.Hkv + h) * (int64_t)A.D + c * 8;
    *reinterpret_cast<uint4*>(A.k_store + dst) = *reinterpret_cast<const uint4*>(A.k_new + src);
    *reinterpret_cast<uint4*>(A.v_store + dst) = *reinterpret_cast<const uint4*>(A.v_new + src);
  }
}

const void* append_kernel_ptr() { return (const void*)sdpa_append_kernel; }

}  // namespace sdpa
