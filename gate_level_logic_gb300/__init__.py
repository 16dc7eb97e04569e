"""GB300-native gate-level re-simulator (GATSPI-style hybrid event/implicit
per-logic-level gate evaluation) on hand-written sm_103a CUDA kernels.

* ``gatspi``    -- ctypes binding of the C ABI (include/gatspi.h), same names;
* ``Simulator`` -- numpy/torch front end over that ABI;
* ``sdf_annotate`` -- SDF text to delay tables through the library's translator;
* ``build``     -- compiles libgatspi.so in-tree.
"""
from . import gatspi  # noqa: F401
from .gatspi import GatspiError  # noqa: F401
from .sdf import sdf_annotate  # noqa: F401
from .simulator import Simulator  # noqa: F401
