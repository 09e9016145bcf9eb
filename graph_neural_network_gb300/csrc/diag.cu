// Self-test of the bounded-wait error path.  One thread waits on an mbarrier
// that no copy and no thread will ever complete; the wait gives up after a
// bounded number of polls, records DEVERR_TIMEOUT in the graph's status word
// and the kernel returns, exactly as a block whose edge-list copy never lands
// does in the aggregation kernels.  Nothing is left in flight: the barrier
// expects an arrival, not a transaction.
#include "device.cuh"

namespace gnn {
namespace {

__global__ void wait_selftest(int polls, int32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival that never comes
    if (!mbar_wait(&bar, 0, polls)) atomicOr(err, DEVERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_wait_selftest(const gnn_graph* g, int polls, cudaStream_t st) {
  wait_selftest<<<1, 32, 0, st>>>(polls, g->err);
  return cudaGetLastError();
}

}  // namespace gnn
