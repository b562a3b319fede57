"""GB300-native (sm_103a) tile-binned Gaussian-splat rasterization.

The compute lives in a C-ABI CUDA library (csrc/, declared in
include/gs_splat.h); `binding` marshals torch tensors to it.  Importing this
package loads nothing; the library is opened on the first call.
"""

__version__ = "0.1.0"
