// decode_bf16.cu -- bf16-cache variants of the main decode kernel.
#include "decode_kernel.cuh"

namespace kvp {

#define KVP_BF16_VARIANTS(X) \
    X(64, 16, 8) X(64, 16, 16) X(64, 32, 8) X(64, 32, 16) \
    X(128, 16, 8) X(128, 16, 16) X(128, 32, 8) X(128, 32, 16)

cudaError_t launch_decode_bf16(int head_dim, int block_size, int head_tile, dim3 grid,
                               const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, cudaStream_t s)
{
#define KVP_CASE(D_, BS_, NT_) \
    if (head_dim == D_ && block_size == BS_ && head_tile == NT_) \
        return launch_variant<false, D_, BS_, NT_>(grid, tk, tv, p, s);
    KVP_BF16_VARIANTS(KVP_CASE)
#undef KVP_CASE
    return cudaErrorInvalidValue;
}

cudaError_t prepare_decode_bf16(int head_dim, int block_size, int head_tile)
{
#define KVP_CASE(D_, BS_, NT_) \
    if (head_dim == D_ && block_size == BS_ && head_tile == NT_) \
        return prepare_variant<false, D_, BS_, NT_>();
    KVP_BF16_VARIANTS(KVP_CASE)
#undef KVP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvp
