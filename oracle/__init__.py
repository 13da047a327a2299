"""CPU oracle (test infrastructure): see ``oracle.mhcpb_oracle``."""
from .mhcpb_oracle import (  # noqa: F401
    N_PROJ, tf32_rna, bf16_bits_to_f64, bf16_bits_to_f32, bf16_rne_from_f64,
    bf16_rne_from_f32, dx_core_f64, dw_f64, add_bf16_like_autograd,
    mhc_proj_rms_backward, bf16_ulp, dx_abs_bound, dw_abs_bound, check_dx, check_dw,
)
