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

namespace sdpa {

// seq_clone ("[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV columns",
// the #24073 commit message in its stack: seq_clone, a device copy of the source prefix).
// Positions [max(0, n - rows), n) of the source column live in store rows [0, min(n, rows)),
// each at row j % rows; they are copied row for row into the destination column, every KV
// head, K and V.  A column's cell of one row is Hkv * D contiguous elements; the grid walks
// 16-byte chunks, four per thread per step so each thread keeps four loads in flight.
__global__ void __launch_bounds__(kCloneThreads) sdpa_clone_kernel(CloneArgs A) {
  const int cpr = A.Hkv * (A.D / 8);  // chunks per (row, column) cell
  const int64_t total = A.m * cpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < total; base += 4 * stride) {
    uint4 kk[4], vv[4];
    int64_t dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t idx = base + u * stride;
      dst[u] = -1;
      if (idx < total) {
        const int64_t r = idx / cpr;
        const int c = (int)(idx - r * cpr);
        const int64_t cell = r * A.cols;
        const int64_t src = (cell + A.src_col) * A.Hkv * A.D + (int64_t)c * 8;
        dst[u] = (cell + A.dst_col) * A.Hkv * A.D + (int64_t)c * 8;
        kk[u] = *reinterpret_cast<const uint4*>(A.k_store + src);
        vv[u] = *reinterpret_cast<const uint4*>(A.v_store + src);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (dst[u] < 0) continue;
      *reinterpret_cast<uint4*>(A.k_store + dst[u]) = kk[u];
      *reinterpret_cast<uint4*>(A.v_store + dst[u]) = vv[u];
    }
  }
}

const void* clone_kernel_ptr() { return (const void*)sdpa_clone_kernel; }

}  // namespace sdpa
