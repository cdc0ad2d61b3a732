// decode_heads.cu -- variants of the decode kernel whose CTA covers a group of kv heads
// (decode_heads.cuh): the shapes the planner picks with the automatic chunk.
#include "decode_heads.cuh"

namespace kvp {

// (fp8, head_dim, block_size, row tile, kv heads per CTA, CTAs per SM)
#define KVP_HEADS_VARIANTS(X) X(false, 128, 16, 8, 2, 3) X(true, 128, 32, 8, 4, 2)

bool decode_heads_supported(bool fp8, int head_dim, int block_size, int head_tile, int heads,
                            int ctas)
{
#define KVP_CASE(F_, D_, BS_, NT_, HC_, CT_)                                              \
    if (fp8 == F_ && head_dim == D_ && block_size == BS_ && head_tile == NT_ && heads == HC_ && \
        ctas == CT_)                                                                       \
        return true;
    KVP_HEADS_VARIANTS(KVP_CASE)
#undef KVP_CASE
    return false;
}

cudaError_t launch_decode_heads(bool fp8, int head_dim, int block_size, int head_tile, int heads,
                                int ctas, dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv,
                                const DecodeParams& p, cudaStream_t s)
{
#define KVP_CASE(F_, D_, BS_, NT_, HC_, CT_)                                              \
    if (fp8 == F_ && head_dim == D_ && block_size == BS_ && head_tile == NT_ && heads == HC_ && \
        ctas == CT_)                                                                       \
        return launch_heads_variant<F_, D_, BS_, NT_, HC_, CT_>(grid, tk, tv, p, s);
    KVP_HEADS_VARIANTS(KVP_CASE)
#undef KVP_CASE
    return cudaErrorInvalidValue;
}

cudaError_t prepare_decode_heads(bool fp8, int head_dim, int block_size)
{
    cudaError_t e = cudaSuccess;
#define KVP_CASE(F_, D_, BS_, NT_, HC_, CT_)                                 \
    if (e == cudaSuccess && fp8 == F_ && head_dim == D_ && block_size == BS_) \
        e = prepare_heads_variant<F_, D_, BS_, NT_, HC_, CT_>();
    KVP_HEADS_VARIANTS(KVP_CASE)
#undef KVP_CASE
    return e;
}

}  // namespace kvp
