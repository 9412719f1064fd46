// The engine's CUDA-core instantiations (activation codes decoded to fp32,
// paired-FMA dot products) and the launch entry; the engine itself is in
// moeq_stream.cuh.
#include "moeq_stream.cuh"

namespace moeq {

size_t stream_partials_floats(int grid) { return static_cast<size_t>(2) * grid * kMaxTok * kUnitRows; }

cudaError_t launch_stream(const StreamArgs& args, int grid, bool cooperative, cudaStream_t stream) {
    if (args.mma) return launch_stream_mma(args, grid, cooperative, stream);
    return launch_mode<false>(args, grid, cooperative, stream);
}

}  // namespace moeq
