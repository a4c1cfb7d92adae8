// gemv_t3.cu -- streaming GEMV kernel instantiations for T = 3 token columns.
#include "launch_stream.cuh"

namespace qg {
template cudaError_t launch_stream<3, MAXG_SMALL, false, false>(const Params<MAXG_SMALL> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<3, MAXG_SMALL, true, false>(const Params<MAXG_SMALL> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<3, MAXG_SEQ, false, false>(const Params<MAXG_SEQ> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<3, MAXG_SMALL, false, true>(const Params<MAXG_SMALL> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<3, MAXG_SMALL, true, true>(const Params<MAXG_SMALL> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<3, MAXG_SEQ, false, true>(const Params<MAXG_SEQ> &, int, size_t, cudaStream_t, bool);
// the sequence epilogue, on the default path for T = 3 (dp4a)
template cudaError_t launch_stream<3, MAXG_SEQ, false, false, true>(const Params<MAXG_SEQ> &, int, size_t, cudaStream_t, bool);
}  // namespace qg
