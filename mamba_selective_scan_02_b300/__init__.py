"""B300-native Mamba selective scan: a C-ABI CUDA library for sm_103a and a thin
Python binding.  Importing the package loads nothing; the library is opened on
first use and a missing or unloadable library raises."""
