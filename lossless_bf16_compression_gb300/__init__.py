"""GB300-native lossless BF16 exponent codec (ZipCCL-style exponent coding).

``binding`` exposes the C ABI of ``libzc.so`` (``zc_compress``, ``zc_decompress``, ...);
``build`` compiles it for sm_103a; ``workloads`` holds the seeded synthetic inputs.  The
library is loaded on first use and a call fails loudly when it has not been built.
"""
from .binding import (  # noqa: F401
    ZC_BASE_AUTO,
    ZC_ERR_CORRUPT,
    ZC_ERR_CUDA,
    ZC_ERR_INVALID_ARG,
    ZC_ERR_MISALIGNED,
    ZC_ERR_SIZE_MISMATCH,
    ZC_ERR_TIMEOUT,
    ZC_OK,
    ZcError,
    compress,
    decompress,
    status,
    zc_compress,
    zc_decompress,
    zc_max_compressed_bytes,
    zc_max_stream_bytes,
    zc_status,
)
