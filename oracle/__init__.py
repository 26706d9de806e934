"""CPU oracle (test infrastructure only; never imported by the product path)."""
from .qkvp_oracle import *  # noqa: F401,F403
from .qkvp_oracle import (e4m3_decode, e4m3_encode, scale_of, quantize,  # noqa: F401
                          quantize_with_scale, dequantize, packed_width,
                          split_columns, quantize_bank, rope_angles, rope,
                          rope_inverse, rms_norm, packed_gemm, forward,
                          norm_rope_backward, epilogue_backward, grad_gemms,
                          backward, E4M3_MAX)
from .oproj_oracle import (quantize_weight, oproj_forward, oproj_grad_gemms,  # noqa: F401
                           oproj_backward)
from .mlp_oracle import (to_bf16, mlp_forward, mlp_dpre, mlp_grad_gemms,  # noqa: F401
                         mlp_backward)
