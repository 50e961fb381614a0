"""B300-native selective state-space scan (Mamba S6): C-ABI library + thin Python binding.

``selective_state_space_153_b300.ssm`` binds the CUDA library (libssm_scan.so) with
ctypes; ``selective_state_space_153_b300.gen`` makes seeded synthetic inputs. Importing
the package loads neither the CUDA library nor torch's CUDA runtime.
"""
__all__ = ["gen", "ssm"]
