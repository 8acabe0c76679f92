"""FP8 (e4m3fn) W8A8 linear with dynamic per-tensor activation quantization, for sm_103a.

Placeholder binding; the C-ABI library and its loader follow.
"""


def min_ld(K: int) -> int:
    """Leading dimension (bytes) of the library's FP8 matrices: K rounded up to 16."""
    return (int(K) + 15) // 16 * 16
