"""Oracle: FNUZ -> OCP re-encoding of E4M3 bytes (test infrastructure only).

The two dialects share the bit layout and differ by one in the exponent
bias, so a byte read under the wrong dialect is exactly 2x off ("Real-time
VLA inference on AMD hardware", section "Different FP8 representation";
"Deploying DeepSeek-V4-Flash on AMD MI300X", section "The FP8 dialect
problem").  Weights imported in FNUZ are re-encoded so that each byte keeps
its value under OCP.

Readings:
  * value-preserving means exact wherever OCP can hold the FNUZ value and
    round-to-nearest-even otherwise: the re-encode is Encode_OCP of
    Decode_FNUZ.  Eight magnitudes at the bottom of the FNUZ range (exponent
    field 0 or 1 with an odd mantissa) lie halfway between OCP codes and
    round to the even one; a negative value that rounds to zero keeps its
    sign (OCP 0x80).
  * the FNUZ NaN 0x80 maps to the OCP NaN 0x7F.
"""
import numpy as np

from . import e4m3


def fnuz_to_ocp_byte(b):
    """OCP byte holding the value of FNUZ byte ``b``."""
    return e4m3.encode_value(e4m3.decode_byte(b, e4m3.FNUZ), e4m3.OCP)


def fnuz_to_ocp_table():
    """uint8 array of 256 entries: the OCP byte of every FNUZ byte."""
    return np.array([fnuz_to_ocp_byte(b) for b in range(256)], dtype=np.uint8)


_TABLE = None


def fnuz_to_ocp(data):
    """Re-encode an array of FNUZ bytes to OCP bytes."""
    global _TABLE
    if _TABLE is None:
        _TABLE = fnuz_to_ocp_table()
    return _TABLE[np.asarray(data, dtype=np.uint8)]
