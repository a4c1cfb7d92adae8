// gemv_t8.cu -- streaming GEMV kernel instantiations for T = 8 token columns.
#include "launch_stream.cuh"

namespace qg {
template cudaError_t launch_stream<8, MAXG_SMALL, false, false>(const Params<MAXG_SMALL> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<8, MAXG_SMALL, true, false>(const Params<MAXG_SMALL> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<8, MAXG_SEQ, false, false>(const Params<MAXG_SEQ> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<8, MAXG_SMALL, false, true>(const Params<MAXG_SMALL> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<8, MAXG_SMALL, true, true>(const Params<MAXG_SMALL> &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_stream<8, MAXG_SEQ, false, true>(const Params<MAXG_SEQ> &, int, size_t, cudaStream_t, bool);
// the sequence epilogue, on the default path for T = 8 (tensor cores)
template cudaError_t launch_stream<8, MAXG_SEQ, false, true, true>(const Params<MAXG_SEQ> &, int, size_t, cudaStream_t, bool);
}  // namespace qg
