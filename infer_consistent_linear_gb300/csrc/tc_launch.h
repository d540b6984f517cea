// Host entry points of the TC_BF16X3 kernels (defined in tc_launch.cu).
#pragma once
#include <cuda_runtime.h>

#include "tc_bwd.cuh"

namespace cpr {
namespace tc {
struct TcDecArgs;
}
// setup must already have run on `st`; a.dvs selects the state-pass split width.
cudaError_t tc_forward(const tc::TcArgs& a, int64_t cmax, int n_seq, int H, cudaStream_t st);
cudaError_t tc_decode_step(const tc::TcDecArgs& a, int dvs, cudaStream_t st);
// Reading-B decode commit: prep and state pass over a batch of one full chunk per
// sequence, run only for the sequences whose position is 0 (a.commit_pos, a.commit_header
// set); persistent grids of one CTA per SM, each leaving at once when none of its
// units commits.
cudaError_t tc_commit(const tc::TcArgs& a, int n_seq, int H, cudaStream_t st);
// Test support: a bounded mbarrier wait that cannot complete (see cpr_selftest_wait_timeout).
cudaError_t tc_wait_timeout_selftest(uint32_t* err, uint32_t limit, uint32_t* ok_out, cudaStream_t st);
// Training forward (prep + state pass writing the backward's tiles), reverse
// state pass and per-chunk gradients; `f` must have train set and
// blk_bytes = kBlockTrain, `b.ws` the same workspace blocks.  Without
// `recompute` the blocks must already hold a training forward's tiles.
cudaError_t tc_backward(const tc::TcArgs& f, const tc::TcBwdArgs& b, int64_t cmax, int n_seq, int H,
                        cudaStream_t st, bool recompute = true);
}  // namespace cpr
